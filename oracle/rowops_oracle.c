/*
 * rowops oracle: plain, slow, double-precision CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY (see rowops_oracle.h). Written for a reader who
 * checks it against the definitions by eye: one row at a time, the steps in
 * the order the pages give them, plain left-to-right sums in double.
 *
 * Readings where the pages leave a step open (each also listed in the design
 * notes):
 *   - a row whose entries are all -inf has no defined softmax; the pages ask
 *     for an explicit convention [EX §7]. Here it is all zeros.
 *   - a NaN anywhere in a row makes the whole softmax row NaN.
 *   - in the online / split forms a block or chunk with no finite entry has
 *     d = 0 and is skipped when merging, so -inf - (-inf) never occurs.
 *   - the GELU constant is 0.79788456 as printed [KT; 171]; the longer
 *     0.7978845608028654 [FUS §三] differs by < 1e-9 relative.
 */
#include "rowops_oracle.h"

#include <math.h>
#include <stdlib.h>

static const double GELU_SQRT_2_OVER_PI = 0.79788456;
static const double GELU_CUBIC = 0.044715;

double oracle_gelu_sqrt_2_over_pi(void) { return GELU_SQRT_2_OVER_PI; }
double oracle_gelu_cubic(void) { return GELU_CUBIC; }

/* ---------------------------------------------------------------------------
 * Stable softmax [EX §2.4; KT "Triton Softmax"]:
 *   m = max_j x_j ; e_j = exp(x_j - m) ; d = sum_j e_j ; y_j = e_j / d
 * Masked / padding entries are -inf and contribute exp(-inf) = 0 [EX §2.3].
 * ------------------------------------------------------------------------- */
void oracle_softmax_row(const double* x, int64_t n, double* y) {
    double m = -INFINITY;
    int has_nan = 0;
    for (int64_t j = 0; j < n; ++j) {
        if (isnan(x[j])) has_nan = 1;
        else if (x[j] > m) m = x[j];
    }
    if (has_nan) {
        for (int64_t j = 0; j < n; ++j) y[j] = NAN;
        return;
    }
    if (m == -INFINITY) { /* no unmasked entry: convention, all zeros */
        for (int64_t j = 0; j < n; ++j) y[j] = 0.0;
        return;
    }
    double d = 0.0;
    for (int64_t j = 0; j < n; ++j) d += exp(x[j] - m);
    for (int64_t j = 0; j < n; ++j) y[j] = exp(x[j] - m) / d;
}

/* ---------------------------------------------------------------------------
 * Online softmax [EX §2.5; L6 §7.2]. The state is (m, d): the largest entry
 * seen so far and the sum of exp(x - m) over the entries seen so far. For
 * each block B of the row, in order:
 *   m_new = max(m_old, max(B))
 *   d_new = d_old * exp(m_old - m_new) + sum_{x in B} exp(x - m_new)
 * and finally y_j = exp(x_j - m) / d.
 * ------------------------------------------------------------------------- */
void oracle_online_softmax_row(const double* x, int64_t n, int64_t block, double* y, double* m_out,
                               double* d_out) {
    double m = -INFINITY, d = 0.0;
    int has_nan = 0;
    if (block < 1) block = 1;
    for (int64_t start = 0; start < n; start += block) {
        int64_t stop = start + block < n ? start + block : n;
        double bmax = -INFINITY;
        for (int64_t j = start; j < stop; ++j) {
            if (isnan(x[j])) has_nan = 1;
            else if (x[j] > bmax) bmax = x[j];
        }
        if (bmax == -INFINITY) continue; /* block adds nothing to d */
        double m_new = m > bmax ? m : bmax;
        double s = 0.0;
        for (int64_t j = start; j < stop; ++j) s += exp(x[j] - m_new);
        d = d * exp(m - m_new) + s; /* exp(-inf) = 0 on the first block */
        m = m_new;
    }
    if (m_out) *m_out = has_nan ? NAN : m;
    if (d_out) *d_out = has_nan ? NAN : d;
    for (int64_t j = 0; j < n; ++j) {
        if (has_nan) y[j] = NAN;
        else if (d == 0.0) y[j] = 0.0; /* no unmasked entry */
        else y[j] = exp(x[j] - m) / d;
    }
}

/* ---------------------------------------------------------------------------
 * Split-row softmax [EX §2.5 split_online_softmax]: first pass, each chunk c
 * computes its own partial (m_c, d_c) = (max of chunk, sum exp(x - m_c));
 * second pass merges the partials
 *   m = max_c m_c ;  d = sum_c d_c * exp(m_c - m)      (chunks with d_c = 0 skipped)
 * third step writes y_j = exp(x_j - m) / d.
 * ------------------------------------------------------------------------- */
void oracle_split_softmax_row(const double* x, int64_t n, int64_t chunk, double* y, double* m_out,
                              double* d_out) {
    if (chunk < 1) chunk = 1;
    int64_t nchunks = (n + chunk - 1) / chunk;
    double* pm = (double*)malloc(sizeof(double) * (size_t)(nchunks > 0 ? nchunks : 1));
    double* pd = (double*)malloc(sizeof(double) * (size_t)(nchunks > 0 ? nchunks : 1));
    int has_nan = 0;
    /* first pass: independent partials */
    for (int64_t c = 0; c < nchunks; ++c) {
        int64_t start = c * chunk, stop = start + chunk < n ? start + chunk : n;
        double mc = -INFINITY;
        for (int64_t j = start; j < stop; ++j) {
            if (isnan(x[j])) has_nan = 1;
            else if (x[j] > mc) mc = x[j];
        }
        double dc = 0.0;
        if (mc != -INFINITY)
            for (int64_t j = start; j < stop; ++j) dc += exp(x[j] - mc);
        pm[c] = mc;
        pd[c] = dc;
    }
    /* second pass: merge */
    double m = -INFINITY;
    for (int64_t c = 0; c < nchunks; ++c)
        if (pd[c] != 0.0 && pm[c] > m) m = pm[c];
    double d = 0.0;
    for (int64_t c = 0; c < nchunks; ++c)
        if (pd[c] != 0.0) d += pd[c] * exp(pm[c] - m);
    free(pm);
    free(pd);
    if (m_out) *m_out = has_nan ? NAN : m;
    if (d_out) *d_out = has_nan ? NAN : d;
    for (int64_t j = 0; j < n; ++j) {
        if (has_nan) y[j] = NAN;
        else if (d == 0.0) y[j] = 0.0;
        else y[j] = exp(x[j] - m) / d;
    }
}

/* ---------------------------------------------------------------------------
 * LayerNorm [EX §4.1; FUS §三]:
 *   mean = sum(x) / n
 *   var  = sum((x - mean)^2) / n            (biased: unbiased=False in FUS §三)
 *   z    = (x - mean) / sqrt(var + eps) * w + b
 * Only the n real entries take part (padding never enters the variance).
 * ------------------------------------------------------------------------- */
void oracle_layernorm_row(const double* x, const double* w, const double* b, double eps, int64_t n,
                          double* z) {
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j) s += x[j];
    double mean = s / (double)n;
    double q = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double c = x[j] - mean;
        q += c * c;
    }
    double var = q / (double)n;
    double rstd = 1.0 / sqrt(var + eps);
    for (int64_t j = 0; j < n; ++j) {
        double wj = w ? w[j] : 1.0;
        double bj = b ? b[j] : 0.0;
        z[j] = (x[j] - mean) * rstd * wj + bj;
    }
}

/* ---------------------------------------------------------------------------
 * tanh-approximation GELU [KT "Triton GeLU"; EX §3.4; FUS §三]:
 *   g = 0.5 * z * (1 + tanh(0.79788456 * (z + 0.044715 * z^3)))
 * with the mathematical tanh (libm, double).
 * ------------------------------------------------------------------------- */
double oracle_gelu_tanh(double z) {
    double inner = GELU_SQRT_2_OVER_PI * (z + GELU_CUBIC * z * z * z);
    return 0.5 * z * (1.0 + tanh(inner));
}

/* ---------------------------------------------------------------------------
 * d/dz of the tanh-approximation GELU g(z) = 0.5 z (1 + tanh(u)),
 * u = k0 (z + k1 z^3):
 *   g'(z) = 0.5 (1 + tanh(u)) + 0.5 z (1 - tanh(u)^2) k0 (1 + 3 k1 z^2)
 * ------------------------------------------------------------------------- */
double oracle_gelu_tanh_grad(double z) {
    const double u = GELU_SQRT_2_OVER_PI * (z + GELU_CUBIC * z * z * z);
    const double t = tanh(u);
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * GELU_SQRT_2_OVER_PI * (1.0 + 3.0 * GELU_CUBIC * z * z);
}

/* ---------------------------------------------------------------------------
 * Backward of LayerNorm -> affine -> tanh-GELU [FUS §三 FusedLayerNormGELU].
 * The chain rule through the forward: xh = (x - mean) rstd, z = xh w + b,
 * y = g(z). With dz = dy g'(z) and dxh = dz w, and since mean and rstd depend
 * on the whole row (d mean / dx_j = 1/n, d rstd / dx_j = -rstd^3 (x_j - mean) / n
 * for the biased variance),
 *   dx_j = rstd (dxh_j - (1/n) sum_k dxh_k - xh_j (1/n) sum_k dxh_k xh_k)
 *   dw_j += dz_j xh_j,  db_j += dz_j.
 * ------------------------------------------------------------------------- */
void oracle_layernorm_gelu_backward_row(const double* x, const double* dy, const double* w, const double* b,
                                        double eps, int64_t n, double* dx, double* dw, double* db) {
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j) s += x[j];
    const double mean = s / (double)n;
    double q = 0.0;
    for (int64_t j = 0; j < n; ++j) q += (x[j] - mean) * (x[j] - mean);
    const double rstd = 1.0 / sqrt(q / (double)n + eps);
    double a1 = 0.0, a2 = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double xh = (x[j] - mean) * rstd;
        const double wj = w ? w[j] : 1.0, bj = b ? b[j] : 0.0;
        const double dz = dy[j] * oracle_gelu_tanh_grad(xh * wj + bj);
        dw[j] += dz * xh;
        db[j] += dz;
        const double dxh = dz * wj;
        a1 += dxh;
        a2 += dxh * xh;
        dx[j] = dxh; /* finished below */
    }
    for (int64_t j = 0; j < n; ++j) {
        const double xh = (x[j] - mean) * rstd;
        dx[j] = rstd * (dx[j] - a1 / (double)n - xh * a2 / (double)n);
    }
}

/* ---------------------------------------------------------------------------
 * Exact GELU [EX §3.4]: gelu_exact(z) = 0.5 * z * (1 + erf(z / sqrt(2))).
 * 1 + erf(u) is evaluated as erfc(-u) (libm, double): the same function, but
 * for z << 0 the sum 1 + erf cancels (at z = -8 it would be off by ~18%),
 * while erfc(-u) keeps full relative precision.
 * ------------------------------------------------------------------------- */
double oracle_gelu_erf(double z) { return 0.5 * z * erfc(-z / sqrt(2.0)); }

/* LayerNorm -> affine -> GELU, one row [FUS §三 _layer_norm_gelu_kernel]. */
void oracle_layernorm_gelu_row(const double* x, const double* w, const double* b, double eps,
                               int64_t n, double* y) {
    oracle_layernorm_row(x, w, b, eps, n, y);
    for (int64_t j = 0; j < n; ++j) y[j] = oracle_gelu_tanh(y[j]);
}

/* ---------------------------------------------------------------------------
 * Causal mask [EX §5.1 Naive Attention: mask = n <= m, query m sees keys n <= m].
 * Rows stack query blocks of `period` rows (row r is query r mod period);
 * `offset` shifts the diagonal (0: the square causal mask).
 * ------------------------------------------------------------------------- */
int64_t oracle_causal_kept(int64_t r, int64_t n, int64_t period, int64_t offset) {
    int64_t kept = r % period + offset + 1;
    if (kept < 0) kept = 0;
    if (kept > n) kept = n;
    return kept;
}

/* ---------------------------------------------------------------------------
 * RMSNorm [EX §4.2]:
 *   inv_rms = 1 / sqrt(mean(x^2) + eps)        (no mean subtracted)
 *   y       = x * inv_rms * w
 * ------------------------------------------------------------------------- */
void oracle_rmsnorm_row(const double* x, const double* w, double eps, int64_t n, double* y) {
    double q = 0.0;
    for (int64_t j = 0; j < n; ++j) q += x[j] * x[j];
    double inv_rms = 1.0 / sqrt(q / (double)n + eps);
    for (int64_t j = 0; j < n; ++j) {
        double wj = w ? w[j] : 1.0;
        y[j] = x[j] * inv_rms * wj;
    }
}

/* Round to nearest, ties to even, keeping `bits` significant bits (normal
 * range only: the values here are far from overflow and underflow). */
static double round_significand(double v, int bits) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    double m = frexp(v, &e); /* v = m * 2^e, 0.5 <= |m| < 1 */
    return ldexp(nearbyint(ldexp(m, bits)), e - bits);
}

/* The storage types of the operations: fp32 (24 significant bits, a plain
 * conversion to float) and bfloat16 (8 significant bits). */
double oracle_round_to(double v, int storage) {
    if (storage == ORACLE_STORE_F32) return (double)(float)v;
    if (storage == ORACLE_STORE_BF16) return round_significand(v, 8);
    return v;
}

/* ---------------------------------------------------------------------------
 * Fused residual + RMSNorm [EX §4.3]:
 *   residual_out = x + residual
 *   out          = residual_out * rsqrt(mean(residual_out^2) + eps) * w
 * residual_out is an output tensor of the operation's own type, and out is
 * the RMSNorm of that tensor, so s is rounded to the storage type before the
 * norm (fused and unfused then give the same out).
 * ------------------------------------------------------------------------- */
void oracle_residual_rmsnorm_row(const double* x, const double* r, const double* w, double eps, int64_t n,
                                 int storage, double* s_out, double* y) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!s) return;
    for (int64_t j = 0; j < n; ++j) s[j] = oracle_round_to(x[j] + r[j], storage);
    if (s_out)
        for (int64_t j = 0; j < n; ++j) s_out[j] = s[j];
    oracle_rmsnorm_row(s, w, eps, n, y);
    free(s);
}

/* ---------------------------------------------------------------------------
 * Row-batch forms: row r of x starts at x + r*ld; output row r at y + r*N.
 * ------------------------------------------------------------------------- */
static double* widen(const float* src, int64_t n) {
    if (!src) return NULL;
    double* d = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!d) return NULL;
    for (int64_t j = 0; j < n; ++j) d[j] = (double)src[j];
    return d;
}

static int bad_shape(const float* x, int64_t M, int64_t N, int64_t ld, const double* y) {
    return M < 0 || N < 1 || ld < N || (M > 0 && (!x || !y));
}

int oracle_softmax_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, double* y) {
    if (bad_shape(x, M, N, ld, y)) return -1;
    double* row = (double*)malloc(sizeof(double) * (size_t)N);
    if (!row) return -1;
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t j = 0; j < N; ++j) row[j] = (double)x[r * ld + j];
        oracle_softmax_row(row, N, y + r * N);
    }
    free(row);
    return 0;
}

int oracle_split_softmax_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, int64_t chunk,
                                  double* y) {
    if (bad_shape(x, M, N, ld, y) || chunk < 1) return -1;
    double* row = (double*)malloc(sizeof(double) * (size_t)N);
    if (!row) return -1;
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t j = 0; j < N; ++j) row[j] = (double)x[r * ld + j];
        oracle_split_softmax_row(row, N, chunk, y + r * N, NULL, NULL);
    }
    free(row);
    return 0;
}

static int layernorm_rows(const float* x, const float* w, const float* b, double eps, int64_t M,
                          int64_t N, int64_t ld, double* y, int with_gelu) {
    if (bad_shape(x, M, N, ld, y)) return -1;
    double* row = (double*)malloc(sizeof(double) * (size_t)N);
    double* wd = widen(w, N);
    double* bd = widen(b, N);
    int rc = 0;
    if (!row || (w && !wd) || (b && !bd)) {
        rc = -1;
    } else {
        for (int64_t r = 0; r < M; ++r) {
            for (int64_t j = 0; j < N; ++j) row[j] = (double)x[r * ld + j];
            if (with_gelu) oracle_layernorm_gelu_row(row, wd, bd, eps, N, y + r * N);
            else oracle_layernorm_row(row, wd, bd, eps, N, y + r * N);
        }
    }
    free(row);
    free(wd);
    free(bd);
    return rc;
}

int oracle_layernorm_gelu_rows_f32(const float* x, const float* w, const float* b, double eps,
                                   int64_t M, int64_t N, int64_t ld, double* y) {
    return layernorm_rows(x, w, b, eps, M, N, ld, y, 1);
}

int oracle_layernorm_rows_f32(const float* x, const float* w, const float* b, double eps, int64_t M,
                              int64_t N, int64_t ld, double* y) {
    return layernorm_rows(x, w, b, eps, M, N, ld, y, 0);
}

int oracle_rmsnorm_rows_f32(const float* x, const float* w, double eps, int64_t M, int64_t N, int64_t ld,
                            double* y) {
    if (bad_shape(x, M, N, ld, y)) return -1;
    double* row = (double*)malloc(sizeof(double) * (size_t)N);
    double* wd = widen(w, N);
    int rc = 0;
    if (!row || (w && !wd)) {
        rc = -1;
    } else {
        for (int64_t r = 0; r < M; ++r) {
            for (int64_t j = 0; j < N; ++j) row[j] = (double)x[r * ld + j];
            oracle_rmsnorm_row(row, wd, eps, N, y + r * N);
        }
    }
    free(row);
    free(wd);
    return rc;
}

int oracle_residual_rmsnorm_rows_f32(const float* x, const float* r, const float* w, double eps, int storage,
                                     int64_t M, int64_t N, int64_t ld, double* s_out, double* y) {
    if (bad_shape(x, M, N, ld, y) || !r) return -1;
    double* xr = (double*)malloc(sizeof(double) * (size_t)N);
    double* rr = (double*)malloc(sizeof(double) * (size_t)N);
    double* wd = widen(w, N);
    int rc = 0;
    if (!xr || !rr || (w && !wd)) {
        rc = -1;
    } else {
        for (int64_t i = 0; i < M; ++i) {
            for (int64_t j = 0; j < N; ++j) {
                xr[j] = (double)x[i * ld + j];
                rr[j] = (double)r[i * ld + j];
            }
            oracle_residual_rmsnorm_row(xr, rr, wd, eps, N, storage, s_out ? s_out + i * N : NULL, y + i * N);
        }
    }
    free(xr);
    free(rr);
    free(wd);
    return rc;
}

int oracle_softmax_causal_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, int64_t period,
                                   int64_t offset, double* y) {
    if (bad_shape(x, M, N, ld, y) || period < 1) return -1;
    double* row = (double*)malloc(sizeof(double) * (size_t)N);
    if (!row) return -1;
    for (int64_t r = 0; r < M; ++r) {
        const int64_t kept = oracle_causal_kept(r, N, period, offset);
        double* yr = y + r * N;
        for (int64_t j = 0; j < kept; ++j) row[j] = (double)x[r * ld + j];
        if (kept > 0) oracle_softmax_row(row, kept, yr);
        for (int64_t j = kept; j < N; ++j) yr[j] = 0.0;
    }
    free(row);
    return 0;
}

int oracle_layernorm_gelu_erf_rows_f32(const float* x, const float* w, const float* b, double eps, int64_t M,
                                       int64_t N, int64_t ld, double* y) {
    const int rc = layernorm_rows(x, w, b, eps, M, N, ld, y, 0);
    if (rc != 0) return rc;
    for (int64_t i = 0; i < M * N; ++i) y[i] = oracle_gelu_erf(y[i]);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Row-wise sum [EX §2.2]: out[i] = sum_j x[i, j] (padding contributes 0), a
 * plain left-to-right sum in double.
 * ------------------------------------------------------------------------- */
int oracle_row_sum_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, double* out) {
    if (bad_shape(x, M, N, ld, out)) return -1;
    for (int64_t r = 0; r < M; ++r) {
        double s = 0.0;
        for (int64_t j = 0; j < N; ++j) s += (double)x[r * ld + j];
        out[r] = s;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Row-wise max [EX §2.3]: out[i] = max_j x[i, j] (padding is -inf); a NaN in
 * the row makes the result NaN (as for softmax, where it poisons the row).
 * ------------------------------------------------------------------------- */
int oracle_row_max_rows_f32(const float* x, int64_t M, int64_t N, int64_t ld, double* out) {
    if (bad_shape(x, M, N, ld, out)) return -1;
    for (int64_t r = 0; r < M; ++r) {
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            const double v = (double)x[r * ld + j];
            if (isnan(v)) {
                m = NAN;
                break;
            }
            if (v > m) m = v;
        }
        out[r] = m;
    }
    return 0;
}

int oracle_layernorm_gelu_backward_rows_f32(const float* x, const float* dy, const float* w, const float* b,
                                            double eps, int64_t M, int64_t N, int64_t ld, double* dx, double* dw,
                                            double* db) {
    if (bad_shape(x, M, N, ld, dx) || !dy || !dw || !db) return -1;
    double* xr = (double*)malloc(sizeof(double) * (size_t)N);
    double* gr = (double*)malloc(sizeof(double) * (size_t)N);
    double* wd = widen(w, N);
    double* bd = widen(b, N);
    int rc = 0;
    if (!xr || !gr || (w && !wd) || (b && !bd)) {
        rc = -1;
    } else {
        for (int64_t j = 0; j < N; ++j) dw[j] = db[j] = 0.0;
        for (int64_t i = 0; i < M; ++i) {
            for (int64_t j = 0; j < N; ++j) {
                xr[j] = (double)x[i * ld + j];
                gr[j] = (double)dy[i * ld + j];
            }
            oracle_layernorm_gelu_backward_row(xr, gr, wd, bd, eps, N, dx + i * N, dw, db);
        }
    }
    free(xr);
    free(gr);
    free(wd);
    free(bd);
    return rc;
}

/* ---------------------------------------------------------------------------
 * Fused residual + bias + GELU [EX §3.4, "fused residual + bias + GELU"]: the
 * page names the fused kernel but gives no formula; the plain reading is the
 * GELU of the elementwise sum x + b + residual, b broadcast along the rows.
 * The three float inputs add exactly in double (their exponents differ by far
 * less than 53 bits in any test), so no summation order is implied.
 * ------------------------------------------------------------------------- */
int oracle_bias_residual_gelu_rows_f32(const float* x, const float* residual, const float* b, int64_t M,
                                       int64_t N, int64_t ld, int approximate, double* y) {
    if (bad_shape(x, M, N, ld, y) || (approximate != 0 && approximate != 1)) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double s = (double)x[i * ld + j];
            if (b) s += (double)b[j];
            if (residual) s += (double)residual[i * ld + j];
            y[i * N + j] = approximate ? oracle_gelu_tanh(s) : oracle_gelu_erf(s);
        }
    return 0;
}
