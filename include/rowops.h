/*
 * rowops: row-wise reduce-then-normalise kernels for one GB300 GPU (sm_103a).
 *
 * C ABI of librowops.so. Every operation works on an M x N row-major matrix
 * whose rows start `ld` elements apart (ld >= N); x and y share ld. All
 * pointers passed as x, y, w, b and workspace are DEVICE pointers owned by the
 * caller; the library allocates nothing and keeps no state between calls
 * except per-device caches of kernel attributes.
 *
 * Sources (lecture notes on CS336 Lecture 6, "Kernels, Triton"):
 *   [L6]  "第 6 讲：GPU Kernels 与 Triton" (cs336.sjfarm.cc)
 *   [KT]  "CS336 Kernels, Triton" notes (yiwen-cai.github.io)
 *   [EX]  "Triton Kernel 实现练习" (lizn-zn.github.io)
 *   [FUS] "PyTorch 自定义 CUDA 算子与 Triton 编程从 Python 原型到 GPU 极致性能" (ocdem.com)
 *
 * Common conventions
 *   - Asynchronous and stream-ordered: a call validates its arguments, enqueues
 *     its kernel(s) on `stream` (which must belong to the current device;
 *     NULL is the legacy default stream) and returns without synchronising.
 *   - Validation happens before any CUDA runtime call, so invalid arguments
 *     return an error code and launch nothing. M == 0 is a no-op (ROWOPS_OK).
 *   - x and y may be the same pointer (in place). Any other overlap between
 *     the x and y row ranges is rejected with ROWOPS_ERR_INVALID_VALUE.
 *   - Pointers must be aligned to their element size; 16-byte alignment of
 *     rows (x, y 16-byte aligned and ld * element size a multiple of 16)
 *     enables the fastest kernels, other alignments are handled by peeling
 *     each row's unaligned head and tail.
 *   - Accumulation is fp32 for both dtypes; bf16 results are rounded to
 *     nearest even. Reductions use a fixed order, so repeated calls on the
 *     same input give bitwise-identical output.
 *   - Launch failures are reported as ROWOPS_ERR_CUDA (from cudaGetLastError
 *     right after the launch). Errors that occur while a kernel runs surface
 *     at the caller's next synchronisation, as for any CUDA kernel.
 *   - Thread-safe; all entry points may be called from any host thread.
 *
 * Benchmarking knobs (environment; unset = automatic). They are read at the
 * library's first call and kept for the process; rowops_reload_tuning()
 * reads them again (for code that changes them between calls, e.g. tests):
 *   ROWOPS_KERNEL=tma|reg|looped|flat  kernel family: TMA-fed row pipeline, register-resident
 *                                 row groups, or the looped any-N kernels; flat: LayerNorm+GELU
 *                                 by chunks of back-to-back rows (ld == N <= 256, x and y
 *                                 16-byte aligned; the default there when N is not a whole
 *                                 number of 16-byte vectors, N <= 128, or the batch is above
 *                                 32 MiB), other operations as reg
 *   ROWOPS_FORCE_TPR=<16..1024>   threads per row (tma: 64..512; flat: 8, 16, 32); row-group
 *                                 split softmax: 256 = two CTAs of 256 threads per SM (default
 *                                 one of 512)
 *   ROWOPS_FORCE_VPT=<n>          16-byte vectors per thread (reg: 1..4; tma: 1, 2, 3, 4, 8)
 *   ROWOPS_FORCE_LOOPED=1         same as ROWOPS_KERNEL=looped
 *   ROWOPS_RING_BUFFERS=<2..16>   rows in flight per row group of the row pipeline (chunks per
 *                                 CTA of the two-pass split softmax on full chunks, default 3;
 *                                 row-group split softmax: the fewest ring slices per CTA its
 *                                 slice size must allow, default 2)
 *   ROWOPS_ROWS_PER_CTA=<1|2|4|5|8> row groups per CTA of the LayerNorm+GELU and RMSNorm row
 *                                 pipelines (5: LayerNorm+GELU with 128 threads x 8 vectors only)
 *   ROWOPS_ONLINE=two_pass|row_groups|single_read  split-row softmax form. Default (chunk 0):
 *                                 row_groups for batches above 32 MiB of rows of at least
 *                                 256 KiB, else two_pass. row_groups spreads each row over a
 *                                 group of CTAs that keep their slices on chip and exchange
 *                                 the slice partials; single_read gives every CTA a column
 *                                 slice of every row. Both read x once (16-byte aligned rows,
 *                                 a length of whole 16-byte vectors, a cooperative launch;
 *                                 other shapes take two_pass).
 *   ROWOPS_PERSIST_L2=1           single_read staged in L2 instead of shared memory
 *   ROWOPS_PERSIST_LOOKAHEAD=<2k> / ROWOPS_PERSIST_PREFETCH=<n>  its pipeline depths
 *   ROWOPS_CTAS_PER_SM=<k>        persistent grid of k CTAs per SM (0 = occupancy limit,
 *                                 -1 = one CTA per row group, no persistence)
 *   ROWOPS_SCHED=static|dynamic   row schedule of the RMSNorm row pipeline on full rows: static
 *                                 (each row group a fixed share) or dynamic (default: work units
 *                                 taken with cluster launch control)
 *   ROWOPS_UNIT_ROWS=<n>          dynamic schedule: rows per row group in one work unit (default 1)
 *   ROWOPS_BWD_PARTIALS=tmem|registers  LayerNorm+GELU backward on full rows: the per-column dw, db
 *                                 partials in tensor memory (default where a 512-thread CTA of
 *                                 two row groups of 256 threads, or four of 128, covers a row
 *                                 with at most 32 columns a thread) or in registers (one row
 *                                 group of up to 1024 threads per CTA)
 *   ROWOPS_WAIT_LIMIT_NS=<ns>     limit of every device-side wait (default 2 s)
 *   ROWOPS_TEST_STALL_ROW=<row>   test hook for the timeout path: the wait that concerns this
 *                                 row is made to run out (the row pipeline's bulk copy of it is
 *                                 expected to bring 16 bytes more than it does; in the two-pass
 *                                 split softmax on full chunks the same for work item <row>,
 *                                 i.e. chunk (row mod nchunks) of row row / nchunks; in the
 *                                 single-read split softmax CTA 0 withholds that row's partial,
 *                                 in the row-group form the CTA of its first slice does).
 *                                 Nothing faults or hangs: the wait gives up at its limit, the
 *                                 kernel records ROWOPS_ERR_TIMEOUT and returns.
 */
#ifndef ROWOPS_H
#define ROWOPS_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rowops_dtype {
    ROWOPS_F32 = 0,  /* IEEE binary32 in and out */
    ROWOPS_BF16 = 1, /* bfloat16 in and out, fp32 arithmetic inside */
} rowops_dtype_t;

typedef enum rowops_status {
    ROWOPS_OK = 0,
    ROWOPS_ERR_INVALID_VALUE = 1, /* null pointer, bad shape / stride / dtype, misaligned pointer, overlap */
    ROWOPS_ERR_UNSUPPORTED = 2,   /* valid but outside what the library handles (e.g. N >= 2^31) */
    ROWOPS_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or smaller than the query says */
    ROWOPS_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    ROWOPS_ERR_TIMEOUT = 5,       /* a device-side wait gave up (reported by the status query) */
} rowops_status_t;

/* Human-readable name of a status code (static storage, never NULL). */
const char* rowops_status_string(rowops_status_t status);

/*
 * Re-reads the ROWOPS_* benchmarking knobs (listed at the top of this header)
 * from the process environment; later calls use the new values. Without it
 * the knobs are read once, at the first call. No CUDA call; thread-safe.
 * (No counterpart on the source pages: a knob-handling convenience.)
 */
void rowops_reload_tuning(void);

/*
 * Stable softmax of every row [EX §2.4 Softmax; KT "Triton Softmax"]:
 *   m = max_j x[r, j];  y[r, j] = exp(x[r, j] - m) / sum_k exp(x[r, k] - m)
 * -inf entries (masked) produce exactly 0. A row whose entries are all -inf
 * produces all zeros (the pages require an explicit convention, [EX §7]). A NaN
 * anywhere in a row makes that row NaN.
 *
 *   x, y   device pointers to M rows of `ld` elements of `dtype`; y may equal x.
 *   M      rows (>= 0); N columns (1 <= N < 2^31); ld row stride in elements (>= N).
 * In batches above 32 MiB, rows of at least 8 KB (bf16) or 16 KB (fp32) and
 * at most 4096 16-byte vectors whose x and y share their offset modulo 16
 * bytes stream through shared memory: bulk asynchronous copies fill a ring of
 * row buffers while earlier rows are reduced and written (one HBM read, one
 * write). Smaller batches and shorter rows are held in registers by row groups
 * of 16..1024 threads (the faster choice there); longer rows, and x and y at
 * different offsets modulo 16 bytes, use an in-CTA online (m, d) loop that
 * reads the row twice [L6 §7.2]. The other row operations choose the same
 * way, with their own row sizes: 4 KB for LayerNorm+GELU and RMSNorm, 16 KB
 * for row sum and max.
 */
rowops_status_t rowops_softmax(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                               rowops_dtype_t dtype, cudaStream_t stream);

/*
 * Causal softmax [EX §5.1 Naive Attention, causal mask n <= m; EX §2.4 Softmax]:
 * rows stack query blocks of `period` rows; row r is query r mod period and
 * keeps the columns c <= (r mod period) + offset:
 *   kept = clamp((r mod period) + offset + 1, 0, N)
 *   y[r, j] = exp(x[r, j] - m) / sum_{k < kept} exp(x[r, k] - m)   for j < kept
 *   y[r, j] = 0                                                    for j >= kept
 * with m the maximum over the kept columns. The masked columns of x are never
 * read (they may hold anything, NaN included); a row that keeps nothing is all
 * zeros. Within the kept columns the conventions of rowops_softmax hold (-inf
 * entries give 0, a NaN makes the row NaN). rowops_softmax on x with -inf in
 * the masked columns gives the same y while reading every column.
 *
 *   x, y, M, N, ld, dtype, stream   as for rowops_softmax.
 *   period   >= 1 (period == N with offset 0: stacked square causal masks).
 *   offset   shifts the diagonal; |offset| <= 2^62.
 * Full rows (16-byte aligned, N a multiple of the 16-byte vector and of a
 * row-pipeline tile) copy only the 16-byte vectors holding kept columns into
 * the row ring; other layouts take a looped kernel.
 */
rowops_status_t rowops_softmax_causal(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int64_t period,
                                      int64_t offset, rowops_dtype_t dtype, cudaStream_t stream);

/*
 * Row-wise sum and row-wise max [EX §2.2 Row-wise Sum, §2.3 Row-wise Max;
 * KT "Triton Row Sum" for rows longer than one block]:
 *   rowops_row_sum: out[i] = sum_j x[i, j]
 *   rowops_row_max: out[i] = max_j x[i, j]   (a NaN in the row gives NaN)
 * fp32 accumulation; out holds M fp32 results for either input dtype.
 *
 *   x, M, N, ld, dtype, stream   as for rowops_softmax.
 *   out   device pointer to M floats, 4-byte aligned, not overlapping x's rows.
 * Same kernel families as rowops_softmax (row pipeline, register row groups,
 * looped CTA per row), reading every element once.
 */
rowops_status_t rowops_row_sum(const void* x, float* out, int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype,
                               cudaStream_t stream);
rowops_status_t rowops_row_max(const void* x, float* out, int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype,
                               cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error word
 * on the current device. Kernels that wait on asynchronous copies (the TMA-fed
 * row pipeline behind rowops_softmax, rowops_layernorm_gelu and the RMSNorm
 * entry points, and the chunked LayerNorm+GELU of short rows) bound every
 * wait; if one gives up, the kernel stops, records ROWOPS_ERR_TIMEOUT there,
 * and the outputs of that call are unspecified. Returns ROWOPS_OK,
 * ROWOPS_ERR_TIMEOUT, or ROWOPS_ERR_CUDA if a CUDA call fails.
 */
rowops_status_t rowops_device_status(cudaStream_t stream);

/*
 * Bytes of device workspace that rowops_online_softmax needs for an M x N
 * problem (any chunk size the call accepts). Returns 0 for invalid arguments
 * (M < 0, N < 1, bad dtype). Pure host arithmetic; no CUDA call.
 */
size_t rowops_online_softmax_workspace_bytes(int64_t M, int64_t N, rowops_dtype_t dtype);

/*
 * Split-row online softmax [EX §2.5 split_online_softmax; L6 §7.2]: each row is
 * cut into chunks of `chunk` columns handled by different CTAs. A first pass
 * computes every chunk's partial (m_c, d_c) = (max, sum exp(x - m_c)); a second
 * pass merges a row's partials as
 *   m = max_c m_c,   d = sum_c d_c * exp(m_c - m)      (chunks with d_c = 0 skipped)
 * and writes y = exp(x - m) / d. Results equal rowops_softmax up to fp32
 * rounding (independent of the chunk count up to rounding).
 *
 * With chunk 0, batches above 32 MiB of rows of at least 256 KiB run as one
 * cooperative kernel in which every chunk stays on chip between the two
 * passes (x is read once): the CTAs that hold a row's chunks store their
 * partials in the workspace and each merges all of them, in chunk order,
 * before writing its chunk of y. Other shapes, and any nonzero chunk, run as
 * two kernels (partials, then merge + normalise). Both give the same results
 * up to fp32 rounding.
 *
 *   x, y, M, N, ld, dtype   as for rowops_softmax.
 *   workspace   device pointer, 256-byte aligned, at least
 *               rowops_online_softmax_workspace_bytes(M, N, dtype) bytes; the call
 *               overwrites it. Its contents before the call do not matter (the
 *               single-kernel form zeroes the slots it uses itself, so no fill is
 *               enqueued). Calls that share a workspace must be ordered on one
 *               stream.
 *   chunk       columns per chunk: 0 picks one from N and the SM count; otherwise
 *               a multiple of 16 in [256, 2^30]. Larger chunks than N are clamped.
 */
rowops_status_t rowops_online_softmax(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                                      rowops_dtype_t dtype, void* workspace,
                                      size_t workspace_bytes, int64_t chunk,
                                      cudaStream_t stream);

/*
 * Synchronises `stream`, then reads the device-side status word that the last
 * rowops_online_softmax call on `workspace` left: ROWOPS_OK, or
 * ROWOPS_ERR_TIMEOUT if a bounded device-side wait gave up (the output of that
 * call is then unspecified). ROWOPS_ERR_CUDA if the synchronisation or the
 * read fails, ROWOPS_ERR_WORKSPACE for a NULL workspace.
 */
rowops_status_t rowops_online_softmax_status(const void* workspace, cudaStream_t stream);

/*
 * rowops_online_softmax for callers that cannot allocate device memory.
 * (No counterpart on the source pages: this is an interface convenience.)
 *
 * Same operation, arguments and results as rowops_online_softmax, minus the
 * workspace: the chunk partials go to a 1 MiB array of device memory that the
 * library itself owns. Meant for code that only holds x and y -- a plugin that
 * a host framework calls with device pointers but no allocator or workspace
 * hook, or a latency-critical path where a cudaMalloc (which may synchronise
 * the device) cannot be afforded. The call allocates nothing.
 *
 *   x, y, M, N, ld, dtype, chunk, stream   as for rowops_online_softmax.
 * Returns ROWOPS_ERR_WORKSPACE when the problem needs more partials than the
 * array holds: M * nchunks must not exceed 131040 (nchunks = ceil(N / chunk),
 * with chunk as chosen for chunk == 0 or as given).
 *
 * Notes:
 *   - Every GPU that loads the library reserves that 1 MiB until the process
 *     exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, no allocation) with that device current; make that
 *     first call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Calls whose kernels may overlap on the GPU (different streams without
 *     ordering between them) race on it and give wrong results: order them on
 *     one stream or synchronise between them. Nothing in it needs clearing
 *     before a call.
 */
rowops_status_t rowops_online_softmax_noalloc(const void* x, void* y, int64_t M, int64_t N,
                                              int64_t ld, rowops_dtype_t dtype, int64_t chunk,
                                              cudaStream_t stream);

/*
 * Fused LayerNorm -> affine -> tanh-approximation GELU of every row
 * [FUS §三 _layer_norm_gelu_kernel; EX §4.1 LayerNorm; KT "Triton GeLU"]:
 *   mean = sum_j x_j / N;  var = sum_j (x_j - mean)^2 / N      (biased)
 *   z_j  = (x_j - mean) / sqrt(var + eps) * w_j + b_j
 *   y_j  = 0.5 z_j (1 + tanh(0.79788456 (z_j + 0.044715 z_j^3)))
 * The kernels evaluate the last line as z / (1 + exp(-2u)), which is the same
 * function without the overflow of the pages' (e^{2u} - 1) / (e^{2u} + 1) form.
 *
 *   x, y   device pointers as for rowops_softmax; y may equal x.
 *   w, b   device pointers to N entries of `dtype`, or NULL for weight 1 / bias 0
 *          (the pages load absent entries with 1.0 and 0.0).
 *   eps    added to the variance (the pages' default is 1e-5); must be >= 0 and finite.
 * Kernel choice as for rowops_softmax (row pipeline / registers / looped); w and
 * b are staged once per CTA as fp32 in shared memory, and the row pipeline runs
 * up to 8 rows per CTA over that one staging. Short back-to-back rows (ld == N
 * <= 256, x and y 16-byte aligned) whose length is not a whole number of
 * 16-byte vectors (e.g. bf16 N = 127), or is at most 128, or whose batch is
 * above 32 MiB, go by chunks of rows instead: whole chunks move between global
 * and shared memory as bulk copies, and teams of lanes normalise the rows in
 * shared memory (its bounded waits as above).
 */
rowops_status_t rowops_layernorm_gelu(const void* x, void* y, const void* w, const void* b,
                                      float eps, int64_t M, int64_t N, int64_t ld,
                                      rowops_dtype_t dtype, cudaStream_t stream);

/*
 * rowops_layernorm_gelu with the exact GELU [EX §3.4 gelu_exact]:
 *   y_j = 0.5 z_j (1 + erf(z_j / sqrt(2))) = z_j Phi(z_j)
 * (Phi the standard normal CDF), z_j as for rowops_layernorm_gelu. Same
 * arguments, layouts, kernels and conventions.
 */
rowops_status_t rowops_layernorm_gelu_erf(const void* x, void* y, const void* w, const void* b, float eps,
                                          int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype,
                                          cudaStream_t stream);

/*
 * Backward of LayerNorm -> affine -> tanh-GELU (rowops_layernorm_gelu)
 * [FUS §三 FusedLayerNormGELU; the page's own backward is a stated shortcut
 * without the GELU derivative and LayerNorm's mean / variance terms; this is
 * the exact gradient]. Per row, xh = (x - mean) rstd, z = xh w + b,
 * dz = dy g'(z), dxh = dz w:
 *   dx = rstd (dxh - mean(dxh) - xh mean(dxh xh))
 *   dw = sum over the rows of dz xh,   db = sum over the rows of dz
 * The row statistics are recomputed from x. dx in `dtype`; dw, db in fp32
 * (sums over M rows), deterministic (partial sums per CTA, or per row group of a
 * CTA, added in a fixed order).
 *
 *   x, dy    device pointers to M rows of `ld` elements (inputs).
 *   w, b     as for rowops_layernorm_gelu (NULL: 1, 0).
 *   dx       device pointer to M rows of `ld` elements; must not overlap x or dy.
 *   dw, db   device pointers to N floats each, 4-byte aligned, apart.
 *   workspace, workspace_bytes   device memory, 256-byte aligned, at least
 *            rowops_layernorm_gelu_backward_workspace_bytes(M, N, dtype) bytes
 *            (overwritten), apart from dw and db; calls sharing it must be
 *            ordered on one stream. It holds 2 N floats for each of at most
 *            clamp(2^22 / N, 152, 4096) partial slots (32 MiB for N <= 27594).
 * M == 0 writes zeros to dw and db.
 */
size_t rowops_layernorm_gelu_backward_workspace_bytes(int64_t M, int64_t N, rowops_dtype_t dtype);
rowops_status_t rowops_layernorm_gelu_backward(const void* x, const void* dy, const void* w, const void* b,
                                               float eps, void* dx, float* dw, float* db, int64_t M, int64_t N,
                                               int64_t ld, rowops_dtype_t dtype, void* workspace,
                                               size_t workspace_bytes, cudaStream_t stream);

/*
 * Fused residual + bias + GELU [EX §3.4 Approx Activation names "fused residual
 * + bias + GELU" without a formula; the plain reading]:
 *   y[i, j] = GELU(x[i, j] + bias[j] + residual[i, j])
 * with the sum formed in fp32 ((x + bias) + residual) and the GELU exact
 * (approximate == 0, erf) or the tanh form (approximate == 1).
 *
 *   x, y       device pointers to M rows of `ld` elements; y may equal x.
 *   residual   device pointer to M rows of `ld` elements, or NULL (no residual);
 *              y may equal it; any other overlap with y is rejected.
 *   bias       device pointer to N elements of `dtype`, or NULL (no bias); must
 *              not overlap y.
 * Aligned rows (x, residual, y at 16-byte row starts, N a multiple of the
 * 16-byte vector, bias 16-byte aligned) take 16-byte vectors; any other layout
 * goes element by element.
 */
rowops_status_t rowops_bias_residual_gelu(const void* x, const void* residual, const void* bias, void* y,
                                          int64_t M, int64_t N, int64_t ld, int approximate, rowops_dtype_t dtype,
                                          cudaStream_t stream);

/*
 * Elementwise GELU of n contiguous elements [EX §3.4 Approx Activation]:
 *   approximate == 0: y = 0.5 x (1 + erf(x / sqrt(2)))             (exact)
 *   approximate == 1: y = 0.5 x (1 + tanh(0.79788456 (x + 0.044715 x^3)))
 *
 *   x, y   device pointers to n elements of `dtype`; y may equal x, any other
 *          overlap is rejected. n >= 0 (n == 0 is a no-op).
 * fp32 arithmetic; bf16 results rounded to nearest even.
 */
rowops_status_t rowops_gelu(const void* x, void* y, int64_t n, int approximate, rowops_dtype_t dtype,
                            cudaStream_t stream);

/*
 * RMSNorm of every row [EX §4.2 RMSNorm]:
 *   inv_rms = 1 / sqrt(sum_j x_j^2 / N + eps);   y_j = x_j * inv_rms * w_j
 * (no mean is subtracted). fp32 accumulation, results cast back to `dtype`.
 *
 *   x, y   device pointers as for rowops_softmax; y may equal x.
 *   w      device pointer to N entries of `dtype`, or NULL for weight 1.
 *   eps    added to the mean square (the pages give no value; 1e-5, the pages'
 *          LayerNorm default, is the binding's default); must be >= 0 and finite.
 * Kernel choice as for rowops_layernorm_gelu (row pipeline with up to 8 rows
 * per CTA over one fp32 staging of w / register row groups / looped).
 */
rowops_status_t rowops_rmsnorm(const void* x, void* y, const void* w, float eps, int64_t M, int64_t N,
                               int64_t ld, rowops_dtype_t dtype, cudaStream_t stream);

/*
 * Fused residual add + RMSNorm [EX §4.3 Fused Residual RMSNorm]:
 *   residual_out = x + residual
 *   y            = residual_out * rsqrt(mean(residual_out^2) + eps) * w
 * returning both tensors, in one pass (x and residual read once, y and
 * residual_out written once). residual_out is rounded to `dtype` (nearest
 * even) and y is the RMSNorm of that stored residual_out, so the fused call
 * gives the same y as rowops_rmsnorm applied to its own residual_out.
 *
 *   x, residual        device pointers to M rows of `ld` elements (inputs).
 *   y, residual_out    device pointers to M rows of `ld` elements (outputs).
 *   Each output may be one of the inputs (in place: e.g. residual_out ==
 *   residual, y == x) or must not overlap either of them; y and residual_out
 *   must not overlap each other. x and residual may be the same. Other
 *   overlaps are rejected with ROWOPS_ERR_INVALID_VALUE.
 *   w, eps, M, N, ld, dtype, stream    as for rowops_rmsnorm.
 * Rows of all four tensors at the same offset modulo 16 bytes take the row
 * pipeline (both input rows of a ring slot arrive on one mbarrier) or the
 * register kernels; other layouts take the looped kernel.
 */
rowops_status_t rowops_fused_residual_rmsnorm(const void* x, const void* residual, void* y, void* residual_out,
                                              const void* w, float eps, int64_t M, int64_t N, int64_t ld,
                                              rowops_dtype_t dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* ROWOPS_H */
