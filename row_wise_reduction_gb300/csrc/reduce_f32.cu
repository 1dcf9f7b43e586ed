// Row sum / row max kernels instantiated for f32 rows.
#include "reduce_inst.cuh"

namespace rowops {
TmaReduceLaunch reduce_tma_f32(int block_index, int vpt_index, bool full, int op) {
    return reduce_tma_table<float>(block_index, vpt_index, full, op);
}
ReduceLaunch reduce_reg_f32(int tpr_index, int vpt, int op) { return reduce_reg_table<float>(tpr_index, vpt, op); }
ReduceLaunch reduce_looped_f32(int op) {
    return op == 0 ? launch_reduce_looped<float, RowSum> : launch_reduce_looped<float, RowMax>;
}
}  // namespace rowops
