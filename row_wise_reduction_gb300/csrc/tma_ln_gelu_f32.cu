// TMA-fed row-pipeline ln+gelu kernels instantiated for f32 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaLnGeluLaunch ln_gelu_tma_f32(int block_index, int vpt_index, bool full) {
    return ln_gelu_tma_table<float>(block_index, vpt_index, full);
}
}  // namespace rowops
