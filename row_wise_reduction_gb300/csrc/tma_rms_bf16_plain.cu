// Row-pipeline RMSNorm kernels (plain form) instantiated for bf16 rows.
#include "tma_rms_inst.cuh"

namespace rowops {
TmaRmsKernel rms_tma_bf16_plain(int tpr, int vpt, int rows, bool full) {
    return rms_tma_lookup<bf16_t, false>(tpr, vpt, rows, full);
}
}  // namespace rowops
