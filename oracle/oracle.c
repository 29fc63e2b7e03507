/*
 * fp64 CPU oracle for the fused decoder operators -- TEST INFRASTRUCTURE.
 *
 * Only tests, the package smoke check and the benchmark's CPU baseline use
 * this file.  It is the plain definition of each operator, in double
 * precision, one loop per step of the definition, single-threaded, with no
 * blocking, fusion or reordering.  It shares no code with the CUDA path.
 *
 * Sources (the web pages on Liger-Kernel that describe the method):
 *  [P1] "Liger-Kernel核心技术：RollingBuffer与融合算子详解"
 *       (Liger-Kernel core techniques: RollingBuffer and fused operators)
 *  [P2] "Liger-Kernel内核级优化：FlashAttention与RollingBuffer详解"
 *  [P3] "Liger-Kernel底层优化：新一代内核级推理加速引擎介绍"
 *  [P4] "Liger-Kernel加持！ms-swift推理延迟降低至毫秒级"
 * Where the pages leave a step open, the textbook definition of the named
 * operator is taken; each such reading is marked READING.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* exact widening of one stored element to double */
static double ld(const void* p, int dt, int64_t i) {
    if (dt == ORC_F64) return ((const double*)p)[i];
    if (dt == ORC_F32) return (double)((const float*)p)[i];
    uint32_t u = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static void widen(const void* p, int dt, int64_t off, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = ld(p, dt, off + i);
}

static int bad_dt(int dt) { return dt < ORC_F64 || dt > ORC_BF16; }

/* ---------------------------------------------------------------- RMSNorm
 * [P3] section "融合内核是如何工作的？来看一段简化版实现" (how the fused kernel
 * works), the RMSNorm step of the fused RMSNorm + QKV + RoPE kernel: the sum
 * of squares of the row, divided by the hidden size, plus epsilon, under an
 * inverse square root, multiplies the element and the per-feature weight.
 * The epsilon is a parameter here (the listing fixes 1e-6). */
int orc_rmsnorm_fwd(const void* x, const void* w, int dt, int64_t rows, int64_t cols, double eps,
                    double* y, double* rstd) {
    if (!x || !w || !y || rows < 0 || cols <= 0 || bad_dt(dt)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double sum_sq = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double v = ld(x, dt, r * cols + j);
            sum_sq += v * v;
        }
        double inv_rms = 1.0 / sqrt(sum_sq / (double)cols + eps);
        if (rstd) rstd[r] = inv_rms;
        for (int64_t j = 0; j < cols; ++j) y[r * cols + j] = ld(x, dt, r * cols + j) * inv_rms * ld(w, dt, j);
    }
    return 0;
}

/* READING: the pages give no backward.  It is the derivative of the forward
 * above: with g = dy * w and r = 1/sqrt(mean(x^2)+eps), dr/dx_k = -r^3 x_k / H,
 *     dx_k = r g_k - (r^3 / H) x_k sum_j g_j x_j,
 *     dw_j = sum over rows of dy_j x_j r. */
int orc_rmsnorm_bwd(const void* dy, const void* x, const void* w, int dt, int64_t rows, int64_t cols,
                    double eps, double* dx, double* dw) {
    if (!dy || !x || !w || !dx || !dw || rows < 0 || cols <= 0 || bad_dt(dt)) return -1;
    for (int64_t j = 0; j < cols; ++j) dw[j] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        double sum_sq = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double v = ld(x, dt, r * cols + j);
            sum_sq += v * v;
        }
        double rr = 1.0 / sqrt(sum_sq / (double)cols + eps);
        double gx = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            gx += ld(dy, dt, r * cols + j) * ld(w, dt, j) * ld(x, dt, r * cols + j);
        for (int64_t j = 0; j < cols; ++j) {
            double xj = ld(x, dt, r * cols + j), dyj = ld(dy, dt, r * cols + j);
            double gj = dyj * ld(w, dt, j);
            dx[r * cols + j] = rr * gj - (rr * rr * rr / (double)cols) * xj * gx;
            dw[j] += dyj * xj * rr;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------- RoPE
 * [P1] section "算子融合" (operator fusion), FusedRoPE paragraph: the rotation
 * angle of each feature pair comes from the token position, generated from
 * the thread index with no stored table.  [P3] fused-kernel listing, RoPE
 * step: feature f is paired by f mod (head_dim/2), i.e. the pairs are
 * (i, i + D/2), the two halves acting as real and imaginary parts.
 * READING: the pages give no frequency schedule; the standard one is taken,
 * phi(p, i) = p * theta^(-2i/D).  The listing's rotation mixes k with v and
 * has no position term; it is read only for the pairing.
 * Forward rotates by +phi, backward (the transpose of an orthogonal map) by
 * -phi. */
int orc_rope(const void* t, int dt, const int32_t* pos, int64_t B, int64_t S, int64_t NH, int64_t D,
             double theta, int sign, double* out) {
    if (!t || !out || B < 0 || S < 0 || NH < 0 || D <= 0 || (D % 2) || bad_dt(dt) || theta <= 0.0) return -1;
    if (sign != 1 && sign != -1) return -1;
    const int64_t half = D / 2;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t s = 0; s < S; ++s) {
            double p = pos ? (double)pos[b * S + s] : (double)s;
            for (int64_t h = 0; h < NH; ++h) {
                int64_t base = ((b * S + s) * NH + h) * D;
                for (int64_t i = 0; i < half; ++i) {
                    double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
                    double phi = (double)sign * p * inv_freq;
                    double c = cos(phi), sn = sin(phi);
                    double a = ld(t, dt, base + i), bb = ld(t, dt, base + i + half);
                    out[base + i] = a * c - bb * sn;
                    out[base + i + half] = bb * c + a * sn;
                }
            }
        }
    return 0;
}

/* RoPE variants (the pages' listing pairs halves; the interleaved pairing
 * (2i, 2i+1) and caller-supplied cos/sin tables are the other conventions in
 * use).  Same rotation, written out per pair. */
int orc_rope_ex(const void* t, int dt, const int32_t* pos, int64_t B, int64_t S, int64_t NH, int64_t D,
                double theta, int sign, int pairing, const double* cos_tab, const double* sin_tab, int64_t n_tab,
                double* out) {
    if (!t || !out || B < 0 || S < 0 || NH < 0 || D <= 0 || (D % 2) || bad_dt(dt)) return -1;
    if ((sign != 1 && sign != -1) || (pairing != 0 && pairing != 1)) return -1;
    if ((cos_tab == NULL) != (sin_tab == NULL)) return -1;
    if (!cos_tab && !(theta > 0.0)) return -1;
    const int64_t half = D / 2;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t s = 0; s < S; ++s) {
            int64_t p = pos ? (int64_t)pos[b * S + s] : s;
            if (cos_tab && (p < 0 || p >= n_tab)) return -2;
            for (int64_t h = 0; h < NH; ++h) {
                int64_t base = ((b * S + s) * NH + h) * D;
                for (int64_t i = 0; i < half; ++i) {
                    double c, sn;
                    if (cos_tab) {
                        c = cos_tab[p * half + i];
                        sn = (double)sign * sin_tab[p * half + i];
                    } else {
                        double phi = (double)sign * (double)p * pow(theta, -2.0 * (double)i / (double)D);
                        c = cos(phi);
                        sn = sin(phi);
                    }
                    int64_t ia = pairing ? base + 2 * i : base + i;
                    int64_t ib = pairing ? base + 2 * i + 1 : base + i + half;
                    double a = ld(t, dt, ia), bb = ld(t, dt, ib);
                    out[ia] = a * c - bb * sn;
                    out[ib] = bb * c + a * sn;
                }
            }
        }
    return 0;
}

/* ------------------------------------------- fused RMSNorm + QKV + RoPE
 * [P3] section "融合内核是如何工作的？来看一段简化版实现": one kernel takes the
 * hidden row through three steps, with nothing written in between:
 *   1. RMSNorm of the row: inv_rms = 1/sqrt(sum_sq / H + eps), and each
 *      normalised feature x_i * inv_rms * w_i (kept in full precision);
 *   2. the Q, K and V projections of the normalised row, each with its bias
 *      (the listing adds q_bias, k_bias, v_bias; NULL here means no bias);
 *   3. RoPE on the projected q and k.
 * READING: the listing's step 3 rotates k against v with no position term
 * (garbled); it is read as the same RoPE as orc_rope -- pairs (i, i + D/2)
 * within every q head and every k head, angle p * theta^(-2i/D), or the
 * caller's cos/sin tables indexed by position -- and v is left unrotated.
 * Weights in nn.Linear layout: Wq [Hq*D, H], Wk and Wv [Hk*D, H].  Outputs
 * q [B,S,Hq,D], k and v [B,S,Hk,D], rstd [B*S] (the inv_rms of each row). */
static void rope_head(double* h, int64_t D, double p, double theta, const double* cos_tab, const double* sin_tab) {
    const int64_t half = D / 2;
    for (int64_t i = 0; i < half; ++i) {
        double c, sn;
        if (cos_tab) {
            c = cos_tab[(int64_t)p * half + i];
            sn = sin_tab[(int64_t)p * half + i];
        } else {
            double phi = p * pow(theta, -2.0 * (double)i / (double)D);
            c = cos(phi);
            sn = sin(phi);
        }
        double a = h[i], b = h[i + half];
        h[i] = a * c - b * sn;
        h[i + half] = b * c + a * sn;
    }
}

int orc_rmsnorm_qkv_rope(const void* x, const void* w, const void* Wq, const void* Wk, const void* Wv,
                         const void* bq, const void* bk, const void* bv, int dt, const int32_t* pos,
                         const double* cos_tab, const double* sin_tab, int64_t n_tab, int64_t B, int64_t S,
                         int64_t H, int64_t Hq, int64_t Hk, int64_t D, double eps, double theta, double* q,
                         double* k, double* v, double* rstd) {
    if (!x || !w || !Wq || !Wk || !Wv || !q || !k || !v || B < 0 || S < 0 || H <= 0 || Hq < 0 || Hk < 0 ||
        D <= 0 || (D % 2) || bad_dt(dt))
        return -1;
    if ((cos_tab == NULL) != (sin_tab == NULL) || (!cos_tab && !(theta > 0.0))) return -1;
    const int64_t nq = Hq * D, nk = Hk * D;
    double* xn = (double*)malloc(sizeof(double) * (size_t)H);
    if (!xn) return -3;
    for (int64_t t = 0; t < B * S; ++t) {
        const int64_t s = t % S;
        const int64_t p = pos ? (int64_t)pos[t] : s;
        if (cos_tab && (p < 0 || p >= n_tab)) {
            free(xn);
            return -2;
        }
        /* 1. RMSNorm */
        double sum_sq = 0.0;
        for (int64_t i = 0; i < H; ++i) {
            double val = ld(x, dt, t * H + i);
            sum_sq += val * val;
        }
        const double inv_rms = 1.0 / sqrt(sum_sq / (double)H + eps);
        if (rstd) rstd[t] = inv_rms;
        for (int64_t i = 0; i < H; ++i) xn[i] = ld(x, dt, t * H + i) * inv_rms * ld(w, dt, i);
        /* 2. projections with bias */
        for (int64_t f = 0; f < nq; ++f) {
            double acc = bq ? ld(bq, dt, f) : 0.0;
            for (int64_t i = 0; i < H; ++i) acc += xn[i] * ld(Wq, dt, f * H + i);
            q[t * nq + f] = acc;
        }
        for (int64_t f = 0; f < nk; ++f) {
            double acck = bk ? ld(bk, dt, f) : 0.0, accv = bv ? ld(bv, dt, f) : 0.0;
            for (int64_t i = 0; i < H; ++i) {
                acck += xn[i] * ld(Wk, dt, f * H + i);
                accv += xn[i] * ld(Wv, dt, f * H + i);
            }
            k[t * nk + f] = acck;
            v[t * nk + f] = accv;
        }
        /* 3. RoPE on every q head and every k head */
        for (int64_t h = 0; h < Hq; ++h) rope_head(q + t * nq + h * D, D, (double)p, theta, cos_tab, sin_tab);
        for (int64_t h = 0; h < Hk; ++h) rope_head(k + t * nk + h * D, D, (double)p, theta, cos_tab, sin_tab);
    }
    free(xn);
    return 0;
}

/* ----------------------------------------------------------------- SwiGLU
 * [P1] section "算子融合", FusedLinearSwiGLU paragraph: the SiLU activation of
 * the gate branch times the up branch, elementwise.  silu(g) = g * sigmoid(g).
 * READING: the backward is the textbook derivative,
 *     du = dy * silu(g),  dg = dy * u * s * (1 + g (1 - s)),  s = sigmoid(g). */
static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

int orc_swiglu_fwd(const void* g, const void* u, int dt, int64_t n, double* y) {
    if (!g || !u || !y || n < 0 || bad_dt(dt)) return -1;
    for (int64_t i = 0; i < n; ++i) {
        double gi = ld(g, dt, i);
        y[i] = gi * sigmoid(gi) * ld(u, dt, i);
    }
    return 0;
}

int orc_swiglu_bwd(const void* dy, const void* g, const void* u, int dt, int64_t n, double* dg, double* du) {
    if (!dy || !g || !u || !dg || !du || n < 0 || bad_dt(dt)) return -1;
    for (int64_t i = 0; i < n; ++i) {
        double gi = ld(g, dt, i), ui = ld(u, dt, i), dyi = ld(dy, dt, i);
        double s = sigmoid(gi);
        du[i] = dyi * gi * s;
        dg[i] = dyi * ui * s * (1.0 + gi * (1.0 - s));
    }
    return 0;
}

/* ------------------------------------------------------ linear + SwiGLU
 * [P1] section "算子融合", FusedLinearSwiGLU paragraph: the gate and up
 * projections of the same input, SiLU of the gate times the up branch.
 * READING: no bias (the page's module is built with bias=False); the
 * backward is the chain rule through the SwiGLU derivative above. */
static double dot_row(const void* A, const void* B, int dt, int64_t a_off, int64_t b_off, int64_t n) {
    double acc = 0.0;
    for (int64_t h = 0; h < n; ++h) acc += ld(A, dt, a_off + h) * ld(B, dt, b_off + h);
    return acc;
}

int orc_linear_swiglu_fwd(const void* X, const void* Wg, const void* Wu, int dt, int64_t T, int64_t H, int64_t I,
                          double* out) {
    if (!X || !Wg || !Wu || !out || T < 0 || H <= 0 || I <= 0 || bad_dt(dt)) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t i = 0; i < I; ++i) {
            double g = dot_row(X, Wg, dt, t * H, i * H, H);
            double u = dot_row(X, Wu, dt, t * H, i * H, H);
            out[t * I + i] = g * sigmoid(g) * u;
        }
    return 0;
}

int orc_linear_swiglu_bwd(const void* X, const void* Wg, const void* Wu, const void* dH, int dt, int64_t T, int64_t H,
                          int64_t I, double* dX, double* dWg, double* dWu) {
    if (!X || !Wg || !Wu || !dH || !dX || !dWg || !dWu || T < 0 || H <= 0 || I <= 0 || bad_dt(dt)) return -1;
    for (int64_t k = 0; k < T * H; ++k) dX[k] = 0.0;
    for (int64_t k = 0; k < I * H; ++k) dWg[k] = dWu[k] = 0.0;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t i = 0; i < I; ++i) {
            double g = dot_row(X, Wg, dt, t * H, i * H, H);
            double u = dot_row(X, Wu, dt, t * H, i * H, H);
            double s = sigmoid(g), d = ld(dH, dt, t * I + i);
            double dg = d * u * s * (1.0 + g * (1.0 - s));
            double du = d * g * s;
            for (int64_t h = 0; h < H; ++h) {
                double x = ld(X, dt, t * H + h);
                dX[t * H + h] += dg * ld(Wg, dt, i * H + h) + du * ld(Wu, dt, i * H + h);
                dWg[i * H + h] += dg * x;
                dWu[i * H + h] += du * x;
            }
        }
    return 0;
}

/* ---------------------------------------------------------- linear + CE
 * [P1] section "算子融合", FusedCrossEntropyLoss paragraph: softmax and the
 * negative log-likelihood are one step taken straight on the classifier-head
 * output, the softmax never being stored.  READING: the classifier head is
 * the linear map z = W x (no bias); the loss of a row is lse(z) - z[label];
 * rows whose label is ignore_index contribute nothing; the mean divides by
 * the count of the other rows (0 when there are none: loss and gradients 0).
 * This is the unchunked definition: one whole row of logits at a time, its
 * maximum, then lse = m + log sum exp(z - m).  No online merge. */
static int64_t count_valid(const int64_t* labels, int64_t T, int64_t V, int64_t ignore_index, int* bad) {
    int64_t n = 0;
    *bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        if (labels[t] == ignore_index) continue;
        if (labels[t] < 0 || labels[t] >= V) *bad = 1;
        ++n;
    }
    return n;
}

/* logits of row t into z[V], returns lse */
static double row_logits(const double* xt, const void* W, int dt, int64_t H, int64_t V, double* z,
                         double* wrow) {
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        widen(W, dt, v * H, H, wrow);
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h) acc += xt[h] * wrow[h];
        z[v] = acc;
        if (acc > m) m = acc;
    }
    double se = 0.0;
    for (int64_t v = 0; v < V; ++v) se += exp(z[v] - m);
    return m + log(se);
}

int orc_linear_ce(const void* X, const void* W, int dt, const int64_t* labels, int64_t T, int64_t H,
                  int64_t V, int64_t ignore_index, int reduction, double grad_scale, double* loss,
                  double* lse, double* dX, double* dW) {
    if (!X || !W || !labels || T < 0 || H <= 0 || V <= 0 || bad_dt(dt) || (reduction != 0 && reduction != 1))
        return -1;
    int bad = 0;
    int64_t n_valid = count_valid(labels, T, V, ignore_index, &bad);
    if (bad) return -5;
    double scale = reduction == 0 ? (n_valid > 0 ? grad_scale / (double)n_valid : 0.0) : grad_scale;
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    double* xt = (double*)malloc(sizeof(double) * (size_t)H);
    double* wrow = (double*)malloc(sizeof(double) * (size_t)H);
    if (!z || !xt || !wrow) {
        free(z); free(xt); free(wrow);
        return -1;
    }
    if (dW) memset(dW, 0, sizeof(double) * (size_t)(V * H));
    double total = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t y = labels[t];
        if (y == ignore_index) {
            if (lse) lse[t] = 0.0;
            if (dX) for (int64_t h = 0; h < H; ++h) dX[t * H + h] = 0.0;
            continue;
        }
        widen(X, dt, t * H, H, xt);
        double l = row_logits(xt, W, dt, H, V, z, wrow);
        if (lse) lse[t] = l;
        total += l - z[y];
        /* D row = scale * (softmax - onehot), kept in z */
        for (int64_t v = 0; v < V; ++v) z[v] = scale * (exp(z[v] - l) - (v == y ? 1.0 : 0.0));
        if (dX) {
            for (int64_t h = 0; h < H; ++h) dX[t * H + h] = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                widen(W, dt, v * H, H, wrow);
                for (int64_t h = 0; h < H; ++h) dX[t * H + h] += z[v] * wrow[h];
            }
        }
        if (dW)
            for (int64_t v = 0; v < V; ++v)
                for (int64_t h = 0; h < H; ++h) dW[v * H + h] += z[v] * xt[h];
    }
    /* the loss itself is not multiplied by grad_scale (the upstream gradient) */
    if (loss) *loss = reduction == 0 ? (n_valid > 0 ? total / (double)n_valid : 0.0) : total;
    free(z); free(xt); free(wrow);
    return 0;
}

int orc_linear_ce_rows(const void* X, const void* W, int dt, const int64_t* labels, int64_t T, int64_t H,
                       int64_t V, int64_t ignore_index, int reduction, double grad_scale,
                       const int64_t* rows, int64_t n_rows, double* lse, double* loss_term, double* dX_rows) {
    if (!X || !W || !labels || !rows || T < 0 || H <= 0 || V <= 0 || bad_dt(dt) ||
        (reduction != 0 && reduction != 1))
        return -1;
    int bad = 0;
    int64_t n_valid = count_valid(labels, T, V, ignore_index, &bad);
    if (bad) return -5;
    double scale = reduction == 0 ? (n_valid > 0 ? grad_scale / (double)n_valid : 0.0) : grad_scale;
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    double* xt = (double*)malloc(sizeof(double) * (size_t)H);
    double* wrow = (double*)malloc(sizeof(double) * (size_t)H);
    if (!z || !xt || !wrow) {
        free(z); free(xt); free(wrow);
        return -1;
    }
    for (int64_t k = 0; k < n_rows; ++k) {
        int64_t t = rows[k];
        if (t < 0 || t >= T) {
            free(z); free(xt); free(wrow);
            return -2;
        }
        int64_t y = labels[t];
        if (y == ignore_index) {
            if (lse) lse[k] = 0.0;
            if (loss_term) loss_term[k] = 0.0;
            if (dX_rows) for (int64_t h = 0; h < H; ++h) dX_rows[k * H + h] = 0.0;
            continue;
        }
        widen(X, dt, t * H, H, xt);
        double l = row_logits(xt, W, dt, H, V, z, wrow);
        if (lse) lse[k] = l;
        if (loss_term) loss_term[k] = l - z[y];
        if (dX_rows) {
            for (int64_t v = 0; v < V; ++v) z[v] = scale * (exp(z[v] - l) - (v == y ? 1.0 : 0.0));
            for (int64_t h = 0; h < H; ++h) dX_rows[k * H + h] = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                widen(W, dt, v * H, H, wrow);
                for (int64_t h = 0; h < H; ++h) dX_rows[k * H + h] += z[v] * wrow[h];
            }
        }
    }
    free(z); free(xt); free(wrow);
    return 0;
}

/* The same definition restricted to the listed vocabulary rows of dW, given
 * every token's lse (as computed above):
 *     dW[v, :] = sum over valid t of scale * (exp(z_t[v] - lse_t) - [y_t = v]) * x_t,
 *     z_t[v] = w_v . x_t.
 * One pass over the tokens per listed row; n_valid (for the mean) is counted
 * over all T labels. */
int orc_linear_ce_dw_rows(const void* X, const void* W, int dt, const int64_t* labels, int64_t T, int64_t H,
                          int64_t V, int64_t ignore_index, int reduction, double grad_scale, const double* lse,
                          const int64_t* vrows, int64_t n_vrows, double* dW_rows) {
    if (!X || !W || !labels || !lse || !vrows || !dW_rows || T < 0 || H <= 0 || V <= 0 || bad_dt(dt) ||
        (reduction != 0 && reduction != 1))
        return -1;
    int bad = 0;
    int64_t n_valid = count_valid(labels, T, V, ignore_index, &bad);
    if (bad) return -5;
    double scale = reduction == 0 ? (n_valid > 0 ? grad_scale / (double)n_valid : 0.0) : grad_scale;
    double* xt = (double*)malloc(sizeof(double) * (size_t)H);
    double* wrow = (double*)malloc(sizeof(double) * (size_t)H);
    if (!xt || !wrow) {
        free(xt); free(wrow);
        return -1;
    }
    for (int64_t k = 0; k < n_vrows; ++k) {
        int64_t v = vrows[k];
        if (v < 0 || v >= V) {
            free(xt); free(wrow);
            return -2;
        }
        widen(W, dt, v * H, H, wrow);
        double* out = dW_rows + k * H;
        for (int64_t h = 0; h < H; ++h) out[h] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t y = labels[t];
            if (y == ignore_index) continue;
            widen(X, dt, t * H, H, xt);
            double z = 0.0;
            for (int64_t h = 0; h < H; ++h) z += wrow[h] * xt[h];
            double d = scale * (exp(z - lse[t]) - (y == v ? 1.0 : 0.0));
            for (int64_t h = 0; h < H; ++h) out[h] += d * xt[h];
        }
    }
    free(xt); free(wrow);
    return 0;
}

