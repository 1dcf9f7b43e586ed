// TMA-fed row-pipeline softmax kernels instantiated for f32 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaSoftmaxLaunch softmax_tma_f32(int block_index, int vpt_index, bool full) {
    return softmax_tma_table<float>(block_index, vpt_index, full);
}
TmaSoftmaxCausalLaunch softmax_tma_causal_f32(int block_index, int vpt_index) {
    return softmax_tma_causal_table<float>(block_index, vpt_index);
}
}  // namespace rowops
