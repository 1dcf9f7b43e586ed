// LayerNorm+GELU (tanh and exact forms) on short back-to-back rows by chunks of
// rows: launch wrapper and the choice of lanes per row.
#include "ln_gelu_flat.cuh"
#include "rowops_launch.h"

namespace rowops {
namespace {

template <typename T, int L, int EPL, bool ERF>
cudaError_t launch_ln_gelu_flat(const void* x, void* y, const void* w, const void* b, float eps, int64_t M,
                                int64_t N, int64_t ld, const LaunchCfg& cfg) {
    (void)ld;  // == N: the caller checks it
    auto kern = ln_gelu_flat_kernel<T, L, EPL, ERF>;
    const int64_t R = flat_chunk_rows(N, Elem<T>::kBytes);
    const size_t smem = kRingHeader + 2 * size_t(R) * size_t(N) * Elem<T>::kBytes;
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), kFlatBlock, smem, (M + R - 1) / R, cfg);
    kern<<<grid, kFlatBlock, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y),
                                                 static_cast<const T*>(w), static_cast<const T*>(b), eps, M, int(N),
                                                 R, cfg.dev_error, cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

// columns per lane for rows of N on L lanes: 4 or 8, the fewer that covers N.
// (16 columns a lane took 75 registers and ran slower than the register-row
// kernel on bf16 65536 x 300 and x 500: 38 and 40 us against 25 and 33.)
template <typename T, int L, bool ERF>
LnGeluLaunch flat_lanes(int64_t N) {
    if (N <= L * 4) return launch_ln_gelu_flat<T, L, 4, ERF>;
    if (N <= L * 8) return launch_ln_gelu_flat<T, L, 8, ERF>;
    return nullptr;
}

// lanes per row: `lanes` if 8, 16 or 32, else the fewest that cover N with at
// most 8 columns each
template <typename T, bool ERF>
LnGeluLaunch flat_for(int64_t N, int lanes) {
    if (lanes == 8) return flat_lanes<T, 8, ERF>(N);
    if (lanes == 16) return flat_lanes<T, 16, ERF>(N);
    if (lanes == 32) return flat_lanes<T, 32, ERF>(N);
    if (N <= 64) return flat_lanes<T, 8, ERF>(N);
    if (N <= 128) return flat_lanes<T, 16, ERF>(N);
    return flat_lanes<T, 32, ERF>(N);
}

}  // namespace

LnGeluLaunch ln_gelu_flat(int es, bool erf, int64_t N, int lanes) {
    if (es == 4) return erf ? flat_for<float, true>(N, lanes) : flat_for<float, false>(N, lanes);
    return erf ? flat_for<bf16_t, true>(N, lanes) : flat_for<bf16_t, false>(N, lanes);
}

}  // namespace rowops
