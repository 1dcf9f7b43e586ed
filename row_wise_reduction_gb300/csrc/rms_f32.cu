// Register-resident and looped RMSNorm kernels instantiated for f32 rows.
#include "rms_inst.cuh"

namespace rowops {
RmsLaunch rms_reg_f32(int tpr_index, int vpt, bool res) { return rms_reg_table<float>(tpr_index, vpt, res); }
RmsLaunch rms_looped_f32(bool res) {
    return res ? launch_rms_looped<float, true> : launch_rms_looped<float, false>;
}
}  // namespace rowops
