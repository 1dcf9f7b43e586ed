// Register-resident and looped RMSNorm kernels instantiated for bf16 rows.
#include "rms_inst.cuh"

namespace rowops {
RmsLaunch rms_reg_bf16(int tpr_index, int vpt, bool res) { return rms_reg_table<bf16_t>(tpr_index, vpt, res); }
RmsLaunch rms_looped_bf16(bool res) {
    return res ? launch_rms_looped<bf16_t, true> : launch_rms_looped<bf16_t, false>;
}
}  // namespace rowops
