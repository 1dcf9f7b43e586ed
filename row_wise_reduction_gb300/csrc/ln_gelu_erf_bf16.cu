// LayerNorm + exact (erf) GELU kernels instantiated for bf16 rows (register-resident
// and looped forms).
#include "ln_gelu_inst.cuh"

namespace rowops {
LnGeluLaunch ln_gelu_erf_reg_bf16(int tpr_index, int vpt, bool aligned) {
    return ln_gelu_reg_table<bf16_t, true>(tpr_index, vpt, aligned);
}
LnGeluLaunch ln_gelu_erf_looped_bf16() { return launch_ln_gelu_looped<bf16_t, true>; }
}  // namespace rowops
