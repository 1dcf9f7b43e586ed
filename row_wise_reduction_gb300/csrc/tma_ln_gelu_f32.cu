// TMA-fed row-pipeline ln+gelu kernels instantiated for f32 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaLnGeluLaunch ln_gelu_tma_f32(int block_index, int vpt_index, bool full) {
    return ln_gelu_tma_table<float>(block_index, vpt_index, full);
}
TmaLnGeluLaunch ln_gelu_tma_multi_f32(int tpr_index, int vpt_index, int rows_index) {
    return ln_gelu_tma_multi_table<float>(tpr_index, vpt_index, rows_index);
}
}  // namespace rowops
