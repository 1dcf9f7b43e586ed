// LayerNorm + exact (erf) GELU kernels instantiated for f32 rows (register-resident
// and looped forms).
#include "ln_gelu_inst.cuh"

namespace rowops {
LnGeluLaunch ln_gelu_erf_reg_f32(int tpr_index, int vpt, bool aligned) {
    return ln_gelu_reg_table<float, true>(tpr_index, vpt, aligned);
}
LnGeluLaunch ln_gelu_erf_looped_f32() { return launch_ln_gelu_looped<float, true>; }
}  // namespace rowops
