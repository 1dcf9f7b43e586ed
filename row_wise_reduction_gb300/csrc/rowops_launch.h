// Host-side glue between the C ABI (rowops_api.cu) and the kernel
// instantiation units. Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace rowops {

// Rows of stride `row_bytes` start at offsets that repeat modulo 16 bytes with
// this period: 16 / gcd(16, row_bytes).
__host__ __device__ constexpr int row_phase_period(int64_t row_bytes) {
    return (row_bytes & 15) == 0 ? 1 : 16 / int(row_bytes & -row_bytes & 15);
}

// The unique id of the CUDA context current on this thread (cuCtxGetId of
// cuCtxGetCurrent, reached through the runtime's driver entry points), 0 when
// no context is current yet. Per-device caches are keyed on it as well as the
// device: after cudaDeviceReset the next context gets a new id, so symbol
// addresses and function attributes are looked up and set again instead of
// reusing values of a context that no longer exists.
unsigned long long current_context_id();

struct LaunchCfg {
    cudaStream_t stream;
    int device;
    unsigned long long ctx = 0;  // current_context_id() of the call
    int num_sms;
    int max_smem_optin;  // bytes of dynamic shared memory a CTA may opt in to
    int ctas_per_sm;     // 0: occupancy limit; -1: one CTA per work item; k > 0: k per SM
    unsigned* dev_error; // the library's device error word on this device (row-pipeline timeouts)
    bool cooperative;    // the device supports cooperative launches
    int persist_lookahead = 0;  // single-read split-row softmax lookahead (0: automatic)
    bool persist_l2 = false;    // single-read split-row softmax staged in L2 instead of shared memory
    int persist_prefetch = 0;   // rows of L2 prefetch ahead (0: automatic)
    unsigned long long wait_ns = 2000000000ull;  // limit of every device-side wait
    int unit_rows = 0;          // full-row pipelines: 0 static schedule, else rows per group in a work
                                // unit taken by cluster launch control
    int64_t stall_row = -1;     // test hook: the row whose wait is made to run out (-1: none)
    int grouped_block = 0;      // row-group split softmax: threads per CTA (0: automatic)
};

// Persistent grid size for `items` independent work items: the occupancy
// limit (or the forced CTAs per SM) times the SM count, capped at `items`.
int grid_for(const void* func, int block, size_t smem, int64_t items, const LaunchCfg& cfg);

// A persistent grid capped at `cap` CTAs per SM unless ROWOPS_CTAS_PER_SM
// chose the count. The one-group row-pipeline kernels hold more CTAs per SM
// than they run best with (a constant named-barrier id leaves the registers
// and shared memory as the only limits); their launchers pass the measured
// best count.
inline int cap_ctas(int grid, int cap, const LaunchCfg& cfg) {
    if (cfg.ctas_per_sm != 0) return grid;
    const int64_t c = int64_t(cap) * cfg.num_sms;
    return grid > c ? int(c) : grid;
}

// CTAs of `func` one SM can hold at once (occupancy API, cached per device).
int ctas_per_sm(const void* func, int block, size_t smem, const LaunchCfg& cfg);

// Allow `func` to use `smem` bytes of dynamic shared memory (once per device).
// max_carveout: also ask for the largest shared-memory carveout (for kernels
// with a small ring per CTA, where the driver's own choice held fewer CTAs per
// SM than the occupancy calculator, which sizes the persistent grid, assumed)
cudaError_t allow_smem(const void* func, size_t smem, const LaunchCfg& cfg, bool max_carveout = false);

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

// TMA-fed row pipeline: one row per CTA of kTmaBlocks[i] threads, kTmaVpts[j]
// vectors per thread; `full` when the row is exactly block * vpt vectors.
constexpr int kTmaBlocks[] = {64, 128, 256, 512};
constexpr int kNumTmaBlocks = 4;
constexpr int kTmaVpts[] = {1, 2, 3, 4, 8};
constexpr int kNumTmaVpts = 5;
constexpr int kTmaRingHeader = 256;
constexpr int kTmaMaxSlots = 32;  // ring slots of all row groups of a CTA (mbarriers in the ring header)
// dynamic schedule: one CTA per work unit of rows_per_cta * unit_rows rows
inline int dyn_grid(int64_t M, int rows_per_cta, int unit_rows) {
    const int64_t unit = int64_t(rows_per_cta) * unit_rows;
    const int64_t g = (M + unit - 1) / unit;
    return int(g < 1 ? 1 : (g > 0x7fffffff ? 0x7fffffff : g));
}

using TmaSoftmaxLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int nbuf,
                                         const LaunchCfg& cfg);
using TmaLnGeluLaunch = cudaError_t (*)(const void* x, void* y, const void* w, const void* b, float eps,
                                        int64_t M, int64_t N, int64_t ld, int nbuf, const LaunchCfg& cfg);
TmaSoftmaxLaunch softmax_tma_f32(int block_index, int vpt_index, bool full);
TmaSoftmaxLaunch softmax_tma_bf16(int block_index, int vpt_index, bool full);
// causal softmax on full rows (row r keeps the columns c <= (r mod period) + offset)
using TmaSoftmaxCausalLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int nbuf,
                                               int64_t period, int64_t offset, const LaunchCfg& cfg);
TmaSoftmaxCausalLaunch softmax_tma_causal_f32(int block_index, int vpt_index);
TmaSoftmaxCausalLaunch softmax_tma_causal_bf16(int block_index, int vpt_index);
using SoftmaxCausalLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                                            int64_t period, int64_t offset, const LaunchCfg& cfg);
SoftmaxCausalLaunch softmax_causal_looped_f32();
SoftmaxCausalLaunch softmax_causal_looped_bf16();

// LayerNorm+GELU instantiations: ROWS = 1 with TPR in kTmaBlocks and VPT in
// kTmaVpts, or several row groups per CTA sharing one staging of w, b with TPR
// in kTmaMultiTpr, VPT in kTmaMultiVpt, ROWS in kTmaMultiRows (at most 512
// threads; 640 for 5 groups of 128 threads x 8 vectors with the tanh GELU, the
// tile of 8192-column bf16 / 4096-column fp32 rows, whose ~96 registers a
// thread fit 640 threads and whose ring and w, b staging fit 5 groups); full
// rows or general rows. Each comes with its launcher
// and a query of how many of its CTAs an SM holds for a given N and ring depth.
constexpr int kTmaMultiTpr[] = {64, 128, 256};
constexpr int kNumTmaMultiTpr = 3;
constexpr int kTmaMultiVpt[] = {2, 4, 8};
constexpr int kNumTmaMultiVpt = 3;
constexpr int kTmaMultiRows[] = {2, 4, 5, 8, 10};
constexpr int kNumTmaMultiRows = 5;
using TmaCtasQuery = int (*)(int64_t N, int nbuf, const LaunchCfg& cfg);
struct TmaLnGeluKernel {
    TmaLnGeluLaunch launch;     // nullptr: no such instantiation
    TmaCtasQuery ctas_per_sm;
};
TmaLnGeluKernel ln_gelu_tma_f32(int tpr, int vpt, int rows, bool full);
TmaLnGeluKernel ln_gelu_tma_bf16(int tpr, int vpt, int rows, bool full);
// the same with the exact (erf) GELU
TmaLnGeluKernel ln_gelu_erf_tma_f32(int tpr, int vpt, int rows, bool full);
TmaLnGeluKernel ln_gelu_erf_tma_bf16(int tpr, int vpt, int rows, bool full);

// RMSNorm / fused residual + RMSNorm: r, ro are the residual input and output
// (NULL in the plain form).
using RmsLaunch = cudaError_t (*)(const void* x, const void* r, void* y, void* ro, const void* w, float eps,
                                  int64_t M, int64_t N, int64_t ld, const LaunchCfg& cfg);
RmsLaunch rms_reg_f32(int tpr_index, int vpt, bool res);
RmsLaunch rms_reg_bf16(int tpr_index, int vpt, bool res);
RmsLaunch rms_looped_f32(bool res);
RmsLaunch rms_looped_bf16(bool res);

// Row-pipeline RMSNorm: TPR in kRmsTpr, VPT in kRmsVpt, ROWS in kRmsRows (TPR *
// ROWS <= 512 unless ROWS = 1), full or general rows, plain or fused form.
constexpr int kRmsTpr[] = {64, 128, 256, 512};
constexpr int kNumRmsTpr = 4;
constexpr int kRmsVpt[] = {1, 2, 4, 8};
constexpr int kNumRmsVpt = 4;
constexpr int kRmsRows[] = {1, 2, 4, 8};
constexpr int kNumRmsRows = 4;
using TmaRmsLaunch = cudaError_t (*)(const void* x, const void* r, void* y, void* ro, const void* w, float eps,
                                     int64_t M, int64_t N, int64_t ld, int nbuf, const LaunchCfg& cfg);
struct TmaRmsKernel {
    TmaRmsLaunch launch;  // nullptr: no such instantiation
    TmaCtasQuery ctas_per_sm;
};
TmaRmsKernel rms_tma_f32_plain(int tpr, int vpt, int rows, bool full);
TmaRmsKernel rms_tma_f32_residual(int tpr, int vpt, int rows, bool full);
TmaRmsKernel rms_tma_bf16_plain(int tpr, int vpt, int rows, bool full);
TmaRmsKernel rms_tma_bf16_residual(int tpr, int vpt, int rows, bool full);
// fp32 w staged by the register kernel: one unused slot per 16-byte vector of columns
inline size_t rms_reg_smem(int64_t N, int es) {
    const int64_t V = 16 / es;
    return size_t(4) * size_t((N + N / V + 4) & ~int64_t(3));
}
// fp32 w staged by the row pipeline: thread-major, + 64 bytes of head/tail weights
inline size_t rms_tma_stage_smem(int block, int vpt, int es, bool full) {
    return size_t(vpt) * block * (16 / es) * 4 + (full ? 0 : 64);
}

// Elementwise GELU on n contiguous elements (erf: exact, else tanh approximation).
using GeluLaunch = cudaError_t (*)(const void* x, void* y, int64_t n, const LaunchCfg& cfg);
GeluLaunch gelu_f32(bool erf);
GeluLaunch gelu_bf16(bool erf);

// y = GELU(x + b + residual) over M rows of stride ld (residual, b may be NULL);
// vec: the 16-byte vector form (aligned rows, N a multiple of the vector).
using BiasResidualGeluLaunch = cudaError_t (*)(const void* x, const void* r, const void* b, void* y, int64_t M,
                                               int64_t N, int64_t ld, const LaunchCfg& cfg);
BiasResidualGeluLaunch bias_residual_gelu_f32(bool erf, bool vec);
BiasResidualGeluLaunch bias_residual_gelu_bf16(bool erf, bool vec);

// LayerNorm -> affine -> tanh-GELU backward: per-CTA dw, db partials (2 N
// floats each, at most bwd_max_partials(N) CTAs) reduced by ln_gelu_bwd_reduce.
// The cap keeps the partials within 32 MiB (at least 152, at most 4096 CTAs).
inline int bwd_max_partials(int64_t N) {
    const int64_t p = (int64_t(1) << 22) / (N > 0 ? N : 1);
    return int(p < 152 ? 152 : (p > 4096 ? 4096 : p));
}
constexpr int kBwdTpr[] = {64, 128, 256, 512, 1024};  // 1024: three-stage kernel only
using TmaBwdLaunch = cudaError_t (*)(const void* x, const void* dy, const void* w, const void* b, float eps,
                                     void* dx, float* part, int64_t M, int64_t N, int64_t ld, int nbuf,
                                     int* grid_out, const LaunchCfg& cfg);
using BwdLaunch = cudaError_t (*)(const void* x, const void* dy, const void* w, const void* b, float eps, void* dx,
                                  float* part, int64_t M, int64_t N, int64_t ld, int* grid_out,
                                  const LaunchCfg& cfg);
// pipe: the three-stage kernel (one reduction per row, nbuf >= 4) instead of
// the one-row-at-a-time kernel (three reductions per row, nbuf >= 2)
TmaBwdLaunch ln_gelu_bwd_tma_f32(int tpr_index, int vpt, bool pipe);
TmaBwdLaunch ln_gelu_bwd_tma_bf16(int tpr_index, int vpt, bool pipe);
// Full rows with the dw, db partials in tensor memory: 512-thread CTAs of
// 512 / tpr row groups (tpr 128 or 256), vpt in {1, 2, 4}; nullptr otherwise.
// grid_out: the partial slots written (CTAs x row groups).
TmaBwdLaunch ln_gelu_bwd_tmem_f32(int tpr, int vpt);
TmaBwdLaunch ln_gelu_bwd_tmem_bf16(int tpr, int vpt);
BwdLaunch ln_gelu_bwd_looped_f32();
BwdLaunch ln_gelu_bwd_looped_bf16();
cudaError_t ln_gelu_bwd_reduce(const float* part, int P, int64_t N, float* dw, float* db, const LaunchCfg& cfg);

// Row sum / row max (op 0 / 1): fp32 results, one per row.
using ReduceLaunch = cudaError_t (*)(const void* x, float* out, int64_t M, int64_t N, int64_t ld,
                                     const LaunchCfg& cfg);
using TmaReduceLaunch = cudaError_t (*)(const void* x, float* out, int64_t M, int64_t N, int64_t ld, int nbuf,
                                        const LaunchCfg& cfg);
TmaReduceLaunch reduce_tma_f32(int block_index, int vpt_index, bool full, int op);
TmaReduceLaunch reduce_tma_bf16(int block_index, int vpt_index, bool full, int op);
ReduceLaunch reduce_reg_f32(int tpr_index, int vpt, int op);
ReduceLaunch reduce_reg_bf16(int tpr_index, int vpt, int op);
ReduceLaunch reduce_looped_f32(int op);
ReduceLaunch reduce_looped_bf16(int op);

// dynamic shared memory of the row-pipeline kernels
inline size_t tma_row_bytes(int64_t N, int es) { return size_t((N * es + 127) / 128 * 128); }
inline size_t tma_ring_smem(int64_t N, int es, int nbuf) { return kTmaRingHeader + size_t(nbuf) * tma_row_bytes(N, es); }
// thread-major fp32 w, b; general rows add 256 bytes for their head/tail columns
inline size_t tma_affine_smem(int block, int vpt, int es, bool full, int64_t /*N*/) {
    return size_t(2) * vpt * block * (16 / es) * 4 + (full ? 0 : 256);
}

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
LnGeluLaunch ln_gelu_erf_reg_f32(int tpr_index, int vpt, bool aligned);
LnGeluLaunch ln_gelu_erf_reg_bf16(int tpr_index, int vpt, bool aligned);
LnGeluLaunch ln_gelu_erf_looped_f32();
LnGeluLaunch ln_gelu_erf_looped_bf16();
// short back-to-back rows (ld == N, N <= kFlatMaxN) by chunks of rows; es: 4
// (fp32) or 2 (bf16); lanes per row 8, 16 or 32 (else automatic); nullptr when
// N is too long for those lanes
constexpr int64_t kFlatMaxN = 256;
LnGeluLaunch ln_gelu_flat(int es, bool erf, int64_t N, int lanes);

SplitLaunch split_softmax_f32();
SplitLaunch split_softmax_bf16();
// The same two passes with the chunks streamed through a ring of `nbuf` slots
// in shared memory (online_softmax_tma.cuh): rows 16-byte aligned, N a
// multiple of the chunk, chunk = 256 threads x 1, 2, 4 or 8 16-byte vectors;
// cudaErrorNotSupported (nothing launched) otherwise.
using SplitTmaLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int64_t chunk,
                                       int64_t nchunks, int nbuf, void* workspace, const LaunchCfg& cfg);
SplitTmaLaunch split_softmax_tma_f32();
SplitTmaLaunch split_softmax_tma_bf16();

// Single-read split-row softmax (persistent cooperative grid); returns
// cudaErrorNotSupported, launching nothing, when the problem does not suit it.
using PersistLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld, void* workspace,
                                      const LaunchCfg& cfg);
PersistLaunch split_persistent_f32();
PersistLaunch split_persistent_bf16();
// Single-read split-row softmax over row groups of CTAs (cooperative grid);
// cudaErrorNotSupported when the shape or device does not suit it.
using GroupedLaunch = cudaError_t (*)(const void* x, void* y, int64_t M, int64_t N, int64_t ld, void* workspace,
                                      int min_buffers, const LaunchCfg& cfg);
GroupedLaunch split_grouped_f32();
GroupedLaunch split_grouped_bf16();
// workspace of the single-read form: header, M row results, M * persistent_slots(N) partials
int64_t persistent_slots(int64_t N);
size_t persistent_rowstat_bytes(int64_t M);
// columns one CTA of the split kernels covers in one unrolled step
int64_t split_step_cols(int elem_bytes);

// Dynamic shared memory the register-resident LN+GELU kernels need for N columns.
// w, b staging of the register kernel: two fp32 arrays of round_up(N, 4) for
// aligned rows, padded (w, b) pairs (9 per 8 columns) otherwise; the larger.
inline size_t ln_gelu_smem_bytes(int64_t N) {
    const size_t columns = size_t(2) * size_t((N + 3) & ~int64_t(3)) * 4;
    const size_t pairs = size_t(8) * size_t(((N + (N >> 3) + 1) + 1) & ~int64_t(1));
    return columns > pairs ? columns : pairs;
}

}  // namespace rowops
