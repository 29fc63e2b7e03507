/*
 * fp64 CPU oracle for the fused decoder operators (test infrastructure only).
 *
 * Plain, single-threaded, unblocked C: each function is the textbook
 * definition of one operator, written out loop by loop, so that it can be
 * checked against the statement of the method by eye.  Inputs are the exact
 * stored values the GPU path reads (float64, float32 or bfloat16 bits),
 * widened exactly to double; results are double.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline call this library.  It shares no code, header or constant with
 * the CUDA implementation.
 */
#ifndef LIGER_ORACLE_H
#define LIGER_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage codes of the input buffers */
enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

/* RMSNorm forward.  y = x * r * w with r = 1/sqrt(mean(x^2) + eps) per row;
 * rstd[row] = r (may be NULL). */
int orc_rmsnorm_fwd(const void* x, const void* w, int dt, int64_t rows, int64_t cols, double eps,
                    double* y, double* rstd);

/* RMSNorm backward, analytic derivative of the forward (r recomputed from x). */
int orc_rmsnorm_bwd(const void* dy, const void* x, const void* w, int dt, int64_t rows, int64_t cols,
                    double eps, double* dx, double* dw);

/* RoPE on t [B, S, NH, D]: pairs (i, i + D/2) rotated by sign * p * theta^(-2i/D),
 * p = pos[b*S + s] or s when pos is NULL.  out may alias nothing; it is
 * written as double [B, S, NH, D]. */
int orc_rope(const void* t, int dt, const int32_t* pos, int64_t B, int64_t S, int64_t NH, int64_t D,
             double theta, int sign, double* out);

/* RoPE variants.  pairing 0: pairs (i, i + D/2); pairing 1: pairs (2i, 2i+1).
 * cos_tab / sin_tab (both NULL, or both given): explicit [n_tab, D/2] tables
 * indexed by position, used instead of theta^(-2i/D) (the sign still applies
 * to the sine). */
int orc_rope_ex(const void* t, int dt, const int32_t* pos, int64_t B, int64_t S, int64_t NH, int64_t D,
                double theta, int sign, int pairing, const double* cos_tab, const double* sin_tab, int64_t n_tab,
                double* out);

/* SwiGLU forward y = silu(g) * u and its backward. */
/* fused RMSNorm + QKV projection (+ bias) + RoPE on q and k, fp64 outputs */
int orc_rmsnorm_qkv_rope(const void* x, const void* w, const void* Wq, const void* Wk, const void* Wv,
                         const void* bq, const void* bk, const void* bv, int dt, const int32_t* pos,
                         const double* cos_tab, const double* sin_tab, int64_t n_tab, int64_t B, int64_t S,
                         int64_t H, int64_t Hq, int64_t Hk, int64_t D, double eps, double theta, double* q,
                         double* k, double* v, double* rstd);

int orc_swiglu_fwd(const void* g, const void* u, int dt, int64_t n, double* y);
int orc_swiglu_bwd(const void* dy, const void* g, const void* u, int dt, int64_t n, double* dg, double* du);

/* FusedLinearSwiGLU: out = silu(X Wg^T) * (X Wu^T), X [T, H], Wg / Wu [I, H];
 * backward from dH [T, I]: dX [T, H], dWg, dWu [I, H]. */
int orc_linear_swiglu_fwd(const void* X, const void* Wg, const void* Wu, int dt, int64_t T, int64_t H, int64_t I,
                          double* out);
int orc_linear_swiglu_bwd(const void* X, const void* Wg, const void* Wu, const void* dH, int dt, int64_t T, int64_t H,
                          int64_t I, double* dX, double* dWg, double* dWu);

/* Linear cross-entropy, unchunked.  z = X W^T; lse; loss over rows with
 * label != ignore_index (mean: divided by their count; sum: not); D = scale *
 * (softmax(z) - onehot), scale = grad_scale / n_valid (mean) or grad_scale
 * (sum), D = 0 on ignored rows; dX = D W, dW = D^T X.  Outputs may be NULL.
 * Returns 0, or -5 for a label outside [0,V) that is not ignore_index. */
int orc_linear_ce(const void* X, const void* W, int dt, const int64_t* labels, int64_t T, int64_t H,
                  int64_t V, int64_t ignore_index, int reduction, double grad_scale, double* loss,
                  double* lse, double* dX, double* dW);

/* The same definition restricted to the listed rows: lse, the per-row loss
 * term (lse - z_label, 0 if ignored) and the dX row, for each listed row.
 * n_valid (for the mean) is counted over all T labels. */
int orc_linear_ce_rows(const void* X, const void* W, int dt, const int64_t* labels, int64_t T, int64_t H,
                       int64_t V, int64_t ignore_index, int reduction, double grad_scale,
                       const int64_t* rows, int64_t n_rows, double* lse, double* loss_term, double* dX_rows);

/* Rows of dW for the listed vocabulary rows, given every token's lse. */
int orc_linear_ce_dw_rows(const void* X, const void* W, int dt, const int64_t* labels, int64_t T, int64_t H,
                          int64_t V, int64_t ignore_index, int reduction, double grad_scale, const double* lse,
                          const int64_t* vrows, int64_t n_vrows, double* dW_rows);

#ifdef __cplusplus
}
#endif
#endif
