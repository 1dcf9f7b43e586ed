// TMA-fed row-pipeline softmax kernels instantiated for bf16 rows.
#include "tma_inst.cuh"

namespace rowops {
TmaSoftmaxLaunch softmax_tma_bf16(int block_index, int vpt_index, bool full) {
    return softmax_tma_table<bf16_t>(block_index, vpt_index, full);
}
TmaSoftmaxCausalLaunch softmax_tma_causal_bf16(int block_index, int vpt_index) {
    return softmax_tma_causal_table<bf16_t>(block_index, vpt_index);
}
}  // namespace rowops
