// Softmax kernels instantiated for fp32 rows.
#include "softmax_inst.cuh"

namespace rowops {
SoftmaxLaunch softmax_reg_f32(int tpr_index, int vpt) { return softmax_reg_table<float>(tpr_index, vpt); }
SoftmaxLaunch softmax_looped_f32() { return launch_softmax_looped<float>; }
SoftmaxCausalLaunch softmax_causal_looped_f32() { return launch_softmax_causal_looped<float>; }
}  // namespace rowops
