// TMA-fed row-pipeline ln+gelu kernels instantiated for bf16 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaLnGeluLaunch ln_gelu_tma_bf16(int block_index, int vpt_index, bool full) {
    return ln_gelu_tma_table<bf16_t>(block_index, vpt_index, full);
}
}  // namespace rowops
