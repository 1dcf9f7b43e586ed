// TMA-fed row-pipeline ln+gelu kernels instantiated for bf16 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaLnGeluKernel ln_gelu_tma_bf16(int tpr, int vpt, int rows, bool full) {
    return ln_gelu_tma_lookup<bf16_t>(tpr, vpt, rows, full);
}
}  // namespace rowops
