// Host-side glue between the C ABI (rowops_api.cu) and the kernel
// instantiation units. Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace rowops {

struct LaunchCfg {
    cudaStream_t stream;
    int device;
    int num_sms;
    int max_smem_optin;  // bytes of dynamic shared memory a CTA may opt in to
    int ctas_per_sm;     // 0: occupancy limit; -1: one CTA per work item; k > 0: k per SM
};

// Persistent grid size for `items` independent work items: the occupancy
// limit (or the forced CTAs per SM) times the SM count, capped at `items`.
int grid_for(const void* func, int block, size_t smem, int64_t items, const LaunchCfg& cfg);

// Allow `func` to use `smem` bytes of dynamic shared memory (once per device).
cudaError_t allow_smem(const void* func, size_t smem, const LaunchCfg& cfg);

// Thread-per-row choices of the register-resident kernels.
constexpr int kTprChoices[] = {16, 32, 64, 128, 256, 512, 1024};
constexpr int kNumTpr = 7;
constexpr int kMaxVpt = 4;

using SoftmaxLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                                      const LaunchCfg& cfg);
using LnGeluLaunch = cudaError_t (*)(const void* x, void* y, const void* w, const void* b,
                                     float eps, int64_t M, int64_t N, int64_t ld,
                                     const LaunchCfg& cfg);
using SplitLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                                    int64_t chunk, int64_t nchunks, void* workspace,
                                    const LaunchCfg& cfg);

// register-resident: tpr_index into kTprChoices, vpt in 1..kMaxVpt
SoftmaxLaunch softmax_reg_f32(int tpr_index, int vpt);
SoftmaxLaunch softmax_reg_bf16(int tpr_index, int vpt);
SoftmaxLaunch softmax_looped_f32();
SoftmaxLaunch softmax_looped_bf16();

// aligned: all rows start on 16-byte boundaries
LnGeluLaunch ln_gelu_reg_f32(int tpr_index, int vpt, bool aligned);
LnGeluLaunch ln_gelu_reg_bf16(int tpr_index, int vpt, bool aligned);
LnGeluLaunch ln_gelu_looped_f32();
LnGeluLaunch ln_gelu_looped_bf16();

SplitLaunch split_softmax_f32();
SplitLaunch split_softmax_bf16();
// columns one CTA of the split kernels covers in one unrolled step
int64_t split_step_cols(int elem_bytes);

// Dynamic shared memory the register-resident LN+GELU kernels need for N columns.
inline size_t ln_gelu_smem_bytes(int64_t N) { return size_t(2) * size_t((N + 3) & ~int64_t(3)) * 4; }

}  // namespace rowops
