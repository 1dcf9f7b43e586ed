// TMA-fed row-pipeline LayerNorm + exact (erf) GELU kernels instantiated for bf16 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaLnGeluKernel ln_gelu_erf_tma_bf16(int tpr, int vpt, int rows, bool full) {
    return ln_gelu_tma_lookup<bf16_t, true>(tpr, vpt, rows, full);
}
}  // namespace rowops
