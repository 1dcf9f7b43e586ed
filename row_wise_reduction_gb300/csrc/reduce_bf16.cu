// Row sum / row max kernels instantiated for bf16 rows.
#include "reduce_inst.cuh"

namespace rowops {
TmaReduceLaunch reduce_tma_bf16(int block_index, int vpt_index, bool full, int op) {
    return reduce_tma_table<bf16_t>(block_index, vpt_index, full, op);
}
ReduceLaunch reduce_reg_bf16(int tpr_index, int vpt, int op) { return reduce_reg_table<bf16_t>(tpr_index, vpt, op); }
ReduceLaunch reduce_looped_bf16(int op) {
    return op == 0 ? launch_reduce_looped<bf16_t, RowSum> : launch_reduce_looped<bf16_t, RowMax>;
}
}  // namespace rowops
