// Softmax kernels instantiated for bf16 rows.
#include "softmax_inst.cuh"

namespace rowops {
SoftmaxLaunch softmax_reg_bf16(int tpr_index, int vpt) { return softmax_reg_table<bf16_t>(tpr_index, vpt); }
SoftmaxLaunch softmax_looped_bf16() { return launch_softmax_looped<bf16_t>; }
SoftmaxCausalLaunch softmax_causal_looped_bf16() { return launch_softmax_causal_looped<bf16_t>; }
}  // namespace rowops
