// Row-pipeline RMSNorm kernels (residual form) instantiated for f32 rows.
#include "tma_rms_inst.cuh"

namespace rowops {
TmaRmsKernel rms_tma_f32_residual(int tpr, int vpt, int rows, bool full) {
    return rms_tma_lookup<float, true>(tpr, vpt, rows, full);
}
}  // namespace rowops
