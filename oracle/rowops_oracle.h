/*
 * rowops oracle: plain, slow, double-precision CPU reference for the row-wise
 * reduce-then-normalise operations (stable softmax, online / split-row
 * softmax, LayerNorm -> affine -> tanh-GELU, RMSNorm and fused residual +
 * RMSNorm).
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the package smoke check and the
 * benchmark's CPU-baseline leg are the only users. The CUDA library never
 * links or calls it, and the two share no code, header or constant.
 *
 * Sources (lecture notes on CS336 Lecture 6, "Kernels, Triton"):
 *   [L6]   "第 6 讲：GPU Kernels 与 Triton" (cs336.sjfarm.cc)
 *   [KT]   "CS336 Kernels, Triton" notes (yiwen-cai.github.io)
 *   [EX]   "Triton Kernel 实现练习" (lizn-zn.github.io)
 *   [171]  "【CS336】lecture6 占用率|bank冲突|Triton|GeLU算子|softmax算子|reduce算子|matmul算子"
 *   [FUS]  "PyTorch 自定义 CUDA 算子与 Triton 编程从 Python 原型到 GPU 极致性能" (ocdem.com)
 *
 * Parity pins: every function here is checked by the CPU test suite against
 * closed forms, invariants, exact-arithmetic brute force and library routines
 * (no function is "parity unpinned").
 */
#ifndef ROWOPS_ORACLE_H
#define ROWOPS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Constants as printed on the pages. */
double oracle_gelu_sqrt_2_over_pi(void); /* 0.79788456  [KT "Triton GeLU"; 171 "GeLU"] */
double oracle_gelu_cubic(void);          /* 0.044715    [KT; EX §3.4; FUS §三] */

/* ---- single rows, double in / double out ---------------------------------- */

/* Stable softmax [EX §2.4; KT "Triton Softmax"]. y may alias x. */
void oracle_softmax_row(const double* x, int64_t n, double* y);

/* Online softmax [EX §2.5; L6 §7.2]: one scan over blocks of `block` entries
 * with the running state (m, d). Writes y and, if non-NULL, the final m, d. */
void oracle_online_softmax_row(const double* x, int64_t n, int64_t block, double* y, double* m_out,
                               double* d_out);

/* Split-row softmax [EX §2.5 split_online_softmax]: per-chunk partials
 * (m_c, d_c) computed independently, merged in a second pass, then every
 * entry normalised with the merged (m, d). */
void oracle_split_softmax_row(const double* x, int64_t n, int64_t chunk, double* y, double* m_out,
                              double* d_out);

/* LayerNorm [EX §4.1; FUS §三]. w, b may be NULL (weight 1, bias 0). */
void oracle_layernorm_row(const double* x, const double* w, const double* b, double eps, int64_t n,
                          double* z);

/* tanh-approximation GELU [KT "Triton GeLU"; EX §3.4; FUS §三]. */
double oracle_gelu_tanh(double z);

/* Exact GELU [EX §3.4]: 0.5 z (1 + erf(z / sqrt(2))), in double (1 + erf(u)
 * evaluated as erfc(-u), without cancellation for z << 0). */
double oracle_gelu_erf(double z);

/* LayerNorm, then affine, then GELU [FUS §三 _layer_norm_gelu_kernel]. */
void oracle_layernorm_gelu_row(const double* x, const double* w, const double* b, double eps,
                               int64_t n, double* y);

/* Columns of row r that a causal mask keeps [EX §5.1: key n is visible to query
 * m when n <= m], for rows that stack query blocks of `period` rows: column c
 * is kept when c <= (r mod period) + offset, so the count is that plus one,
 * clamped to [0, n]. */
int64_t oracle_causal_kept(int64_t r, int64_t n, int64_t period, int64_t offset);

/* RMSNorm [EX §4.2]: inv_rms = 1 / sqrt(mean_j x_j^2 + eps), y_j = x_j * inv_rms * w_j.
 * w may be NULL (weight 1). */
void oracle_rmsnorm_row(const double* x, const double* w, double eps, int64_t n, double* y);

/* Storage types for a value that an operation writes out and then reuses. */
enum { ORACLE_STORE_EXACT = 0, ORACLE_STORE_F32 = 1, ORACLE_STORE_BF16 = 2 };

/* v rounded to nearest (ties to even) in the given storage type. */
double oracle_round_to(double v, int storage);

/* Fused residual + RMSNorm [EX §4.3]: s_j = x_j + r_j, written out in the
 * storage type (rounded to nearest even), and y = RMSNorm(s) of the stored s.
 * s_out may be NULL. */
void oracle_residual_rmsnorm_row(const double* x, const double* r, const double* w, double eps, int64_t n,
                                 int storage, double* s_out, double* y);

/* ---- M rows with a row stride `ld` (elements), output M x N contiguous ------
 * The fp32 forms take inputs already widened to fp32 (bf16 values are exact
 * in fp32) and widen them to double row by row. Return 0, or -1 on bad
 * arguments / allocation failure. */
int oracle_softmax_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, double* y);
int oracle_split_softmax_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, int64_t chunk,
                                  double* y);
int oracle_layernorm_gelu_rows_f32(const float* x, const float* w, const float* b, double eps,
                                   int64_t M, int64_t N, int64_t ld, double* y);
int oracle_layernorm_rows_f32(const float* x, const float* w, const float* b, double eps, int64_t M,
                              int64_t N, int64_t ld, double* y);
int oracle_rmsnorm_rows_f32(const float* x, const float* w, double eps, int64_t M, int64_t N, int64_t ld,
                            double* y);
/* Derivative of the tanh-approximation GELU, d/dz of oracle_gelu_tanh. */
double oracle_gelu_tanh_grad(double z);

/* Backward of LayerNorm -> affine -> tanh-GELU [FUS §三 FusedLayerNormGELU]:
 * the exact gradient of the forward (the page's own backward is a stated
 * shortcut). Per row, with xh = (x - mean) rstd, z = xh w + b:
 *   dz = dy gelu'(z);  dw += dz xh;  db += dz;  dxh = dz w
 *   dx = rstd (dxh - mean(dxh) - xh mean(dxh xh))
 * dx for the row; dw, db ACCUMULATED (callers zero them). w, b may be NULL. */
void oracle_layernorm_gelu_backward_row(const double* x, const double* dy, const double* w, const double* b,
                                        double eps, int64_t n, double* dx, double* dw, double* db);

/* LayerNorm -> affine -> exact (erf) GELU [EX §3.4, §4.1]. */
int oracle_layernorm_gelu_erf_rows_f32(const float* x, const float* w, const float* b, double eps, int64_t M,
                                       int64_t N, int64_t ld, double* y);
/* The backward over M rows of x and dy (same stride): dx (M x N), dw and db
 * (N each) summed over the rows. */
int oracle_layernorm_gelu_backward_rows_f32(const float* x, const float* dy, const float* w, const float* b,
                                            double eps, int64_t M, int64_t N, int64_t ld, double* dx, double* dw,
                                            double* db);
/* Row sum [EX §2.2]: out[i] = sum_j x[i, j], in double. */
int oracle_row_sum_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, double* out);
/* Row max [EX §2.3]: out[i] = max_j x[i, j]; -inf entries are padding; a NaN
 * makes the row's max NaN. */
int oracle_row_max_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, double* out);
/* Causal softmax: the stable softmax of each row's kept prefix (masked
 * entries are not read), 0 on the masked columns. */
int oracle_softmax_causal_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, int64_t period,
                                   int64_t offset, double* y);
/* x and r share the row stride; s_out may be NULL. */
int oracle_residual_rmsnorm_rows_f32(const float* x, const float* r, const float* w, double eps, int storage,
                                     int64_t M, int64_t N, int64_t ld, double* s_out, double* y);

/* Fused residual + bias + GELU [EX §3.4 names it without a formula; reading:
 * y = GELU(x + b + residual), b per column, the sum exact in double].
 * residual (rows of stride ld, like x) and b (N entries) may be NULL;
 * approximate: 0 the exact (erf) GELU, 1 the tanh form. y is M x N. */
int oracle_bias_residual_gelu_rows_f32(const float* x, const float* residual, const float* b, int64_t M,
                                       int64_t N, int64_t ld, int approximate, double* y);

#ifdef __cplusplus
}
#endif
#endif
