// LayerNorm+GELU kernels instantiated for fp32 rows.
#include "ln_gelu_inst.cuh"

namespace rowops {
LnGeluLaunch ln_gelu_reg_f32(int tpr_index, int vpt, bool aligned) {
    return ln_gelu_reg_table<float>(tpr_index, vpt, aligned);
}
LnGeluLaunch ln_gelu_looped_f32() { return launch_ln_gelu_looped<float>; }
}  // namespace rowops
