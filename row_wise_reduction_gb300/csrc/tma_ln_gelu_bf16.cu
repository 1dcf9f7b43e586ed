// TMA-fed row-pipeline ln+gelu kernels instantiated for bf16 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaLnGeluLaunch ln_gelu_tma_bf16(int block_index, int vpt_index, bool full) {
    return ln_gelu_tma_table<bf16_t>(block_index, vpt_index, full);
}
TmaLnGeluLaunch ln_gelu_tma_multi_bf16(int tpr_index, int vpt_index, int rows_index) {
    return ln_gelu_tma_multi_table<bf16_t>(tpr_index, vpt_index, rows_index);
}
}  // namespace rowops
