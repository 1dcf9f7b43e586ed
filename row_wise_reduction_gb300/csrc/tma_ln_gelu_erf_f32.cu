// TMA-fed row-pipeline LayerNorm + exact (erf) GELU kernels instantiated for f32 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaLnGeluKernel ln_gelu_erf_tma_f32(int tpr, int vpt, int rows, bool full) {
    return ln_gelu_tma_lookup<float, true>(tpr, vpt, rows, full);
}
}  // namespace rowops
