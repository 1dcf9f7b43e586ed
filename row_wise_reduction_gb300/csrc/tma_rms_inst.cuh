// Launch wrappers, occupancy queries and the lookup table of the row-pipeline
// RMSNorm kernels for one element type and one form (plain or fused
// residual). Included once per (dtype, form) unit.
#pragma once

#include "rowops_launch.h"
#include "tma_rms_kernels.cuh"

namespace rowops {

template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool RES>
size_t rms_tma_smem(int64_t N, int nbuf) {
    return kRingHeader + size_t(ROWS) * nbuf * (RES ? 2 : 1) * ring_row_bytes(N, Elem<T>::kBytes) +
           rms_stage_bytes<T, TPR, VPT, FULL>();
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool RES>
cudaError_t launch_rms_tma(const void* x, const void* r, void* y, void* ro, const void* w, float eps, int64_t M,
                           int64_t N, int64_t ld, int nbuf, const LaunchCfg& cfg) {
    auto kern = rms_tma_kernel<T, TPR, VPT, ROWS, FULL, RES>;
    const size_t smem = rms_tma_smem<T, TPR, VPT, ROWS, FULL, RES>(N, nbuf);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    const int unit = FULL ? cfg.unit_rows : 0;  // 0: static schedule
    int grid = unit ? dyn_grid(M, ROWS, unit)
                    : grid_for(reinterpret_cast<const void*>(kern), TPR * ROWS, smem, (M + ROWS - 1) / ROWS, cfg);
    if (!unit && ROWS == 1) grid = cap_ctas(grid, 4, cfg);  // one group per CTA: as before the constant barrier id
    if (!FULL) {  // whole phase classes: every class needs a CTA, and they share the grid evenly
        const int period = row_phase_period(ld * int64_t(Elem<T>::kBytes));
        grid = grid >= period ? grid - grid % period : period;
    }
    kern<<<grid, TPR * ROWS, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(r),
                                                 static_cast<T*>(y), static_cast<T*>(ro), static_cast<const T*>(w),
                                                 eps, M, int(N), ld, nbuf, cfg.dev_error, cfg.wait_ns,
                                                 cfg.stall_row, unit);
    return cudaGetLastError();
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool RES>
int ctas_rms_tma(int64_t N, int nbuf, const LaunchCfg& cfg) {
    auto kern = rms_tma_kernel<T, TPR, VPT, ROWS, FULL, RES>;
    const size_t smem = rms_tma_smem<T, TPR, VPT, ROWS, FULL, RES>(N, nbuf);
    if (smem + 1024 > size_t(cfg.max_smem_optin)) return 0;  // 1 KB for the static reduction buffers
    if (allow_smem(reinterpret_cast<const void*>(kern), smem, cfg) != cudaSuccess) {
        cudaGetLastError();  // a candidate that does not fit must not fail the launch that follows
        return 0;
    }
    return ctas_per_sm(reinterpret_cast<const void*>(kern), TPR * ROWS, smem, cfg);
}

// instantiations: TPR in kRmsTpr, VPT in kRmsVpt, ROWS in kRmsRows with
// TPR * ROWS <= 512 (ROWS = 1 at any TPR); full or general rows
template <typename T, int P, int V, int R, bool F, bool RES>
constexpr TmaRmsKernel rms_entry() {
    if constexpr (R == 1 || P * R <= 512)
        return TmaRmsKernel{launch_rms_tma<T, P, V, R, F, RES>, ctas_rms_tma<T, P, V, R, F, RES>};
    else
        return TmaRmsKernel{nullptr, nullptr};
}
#define ROWOPS_RMS3(T, P, V, F, RES) \
    {rms_entry<T, P, V, 1, F, RES>(), rms_entry<T, P, V, 2, F, RES>(), rms_entry<T, P, V, 4, F, RES>(), \
     rms_entry<T, P, V, 8, F, RES>()}
#define ROWOPS_RMS2(T, P, F, RES) \
    {ROWOPS_RMS3(T, P, 1, F, RES), ROWOPS_RMS3(T, P, 2, F, RES), ROWOPS_RMS3(T, P, 4, F, RES), ROWOPS_RMS3(T, P, 8, F, RES)}
#define ROWOPS_RMS1(T, F, RES) \
    {ROWOPS_RMS2(T, 64, F, RES), ROWOPS_RMS2(T, 128, F, RES), ROWOPS_RMS2(T, 256, F, RES), ROWOPS_RMS2(T, 512, F, RES)}

template <int N>
int rms_index_of(const int (&a)[N], int v) {
    for (int i = 0; i < N; ++i)
        if (a[i] == v) return i;
    return -1;
}

template <typename T, bool RES>
TmaRmsKernel rms_tma_lookup(int tpr, int vpt, int rows, bool full) {
    static const TmaRmsKernel tf[kNumRmsTpr][kNumRmsVpt][kNumRmsRows] = ROWOPS_RMS1(T, true, RES);
    static const TmaRmsKernel tg[kNumRmsTpr][kNumRmsVpt][kNumRmsRows] = ROWOPS_RMS1(T, false, RES);
    const int i = rms_index_of(kRmsTpr, tpr), j = rms_index_of(kRmsVpt, vpt), r = rms_index_of(kRmsRows, rows);
    if (i < 0 || j < 0 || r < 0) return TmaRmsKernel{nullptr, nullptr};
    return full ? tf[i][j][r] : tg[i][j][r];
}
#undef ROWOPS_RMS1
#undef ROWOPS_RMS2
#undef ROWOPS_RMS3

}  // namespace rowops
