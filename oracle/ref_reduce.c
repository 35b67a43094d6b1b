/*
 * ref_reduce.c -- CPU oracle for the softmax / LayerNorm reduce path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This file states, as plain and slow
 * double-precision C, what the GPU kernels must compute.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it; the
 * library never does.  It shares no source, header, constant or helper with
 * the CUDA code: the two sides meet only on identical input arrays.
 *
 * Every function follows the plain mathematical definition of the operation
 * (not the fused / rewritten form the kernels use), so that a reader can check
 * it against the sources by eye:
 *
 *   [L10] "CMU 11-868 L10: Accelerating Transformers on GPUs, and Where
 *         LightSeq Finds the Time", section "Technique 2: rewrite the formula,
 *         drop a synchronization" (slides 21-24: LayerNorm statistics, the
 *         LayerNorm backward sums, softmax = max-reduce then exp-sum-reduce).
 *   [HW4] "CMU 11-868 HW4：把 Softmax 與 LayerNorm 寫成 CUDA 融合 kernel",
 *         section 題目結構與配分 (problem structure and grading: Problem 1.1,
 *         future tokens set to -inf, attention mask added, then the row max;
 *         Problem 2.1, sigma = sqrt(mu(x^2) - mu(x)^2 + eps) with eps = 1e-8;
 *         Problem 2.2, an input-gradient kernel and a gamma/beta-gradient
 *         kernel), and section 那些「快幾倍」是跟誰比 (what the speed-ups are
 *         measured against: the test baseline is softmax(inp + mask)).
 *
 * Readings where the sources are silent (each is also listed in the design
 * notes):
 *   - "future tokens" are keys j > query i (causal requires Tq == Tk);
 *   - the additive mask has shape [B, Tk]: one row per batch entry, shared by
 *     every head and every query of that batch entry;
 *   - a row whose every key is masked out produces all zeros (no NaN);
 *   - the variance is the population variance (divide by N), as
 *     mu(x^2) - mu(x)^2 implies, and eps sits inside the square root;
 *   - scores are finite (a masked key contributes exp(-inf) = 0).
 *
 *   [FT]  "FastTransformer: Breaking the Compiler Ceiling via Architectural
 *         Co-Design", section 5.4 "Vectorized Pre-RMSNorm": RMSNorm, the
 *         LayerNorm without mean centring (scale only, no bias).
 *
 *   [L10-T1] the L10 page, section "Technique 1: kernel fusion, leaving only
 *         GEMMs to cuBLAS" (slide 12): cross entropy is the third custom
 *         reduce kernel of the layer, beside LayerNorm and softmax.  The page
 *         gives no formula; the oracle takes the textbook softmax cross
 *         entropy of one target class per row.  Readings: int32 targets; a
 *         negative target marks an ignored (padding) row, whose loss, saved
 *         log-sum-exp and gradient are 0; a target >= V gives NaN loss and
 *         gradient; no label smoothing; one loss per row (the caller
 *         reduces); the backward takes the saved log-sum-exp and a per-row
 *         upstream gradient.
 *
 * Functions take row-major double arrays; the Python wrapper in this package
 * converts the storage-dtype inputs exactly (every fp32/fp16/bf16 value is a
 * double) and rounds nothing on the way in.
 */
#include <math.h>
#include <stdint.h>

/* ------------------------------------------------------------------------ */
/* Attention softmax forward                                                 */
/* ------------------------------------------------------------------------ */
/*
 * For each listed row r (one (batch, head, query) triple of a [B,H,Tq,Tk]
 * score tensor, passed here as its own Tk-long row):
 *   z_j = -inf                       if causal and j > query[r]   [HW4 1.1]
 *   z_j = x_j + mask[batch[r], j]    otherwise (mask may be NULL) [HW4 test]
 *   m   = max_j z_j                  (first reduction, [L10] slide 23)
 *   e_j = exp(z_j - m),  s = sum_j e_j (second reduction)
 *   y_j = e_j / s
 * A row with m = -inf (every key masked) is written as zeros.
 *
 * y, x  : [nrows, Tk]
 * mask  : [B, Tk] or NULL
 * batch : [nrows] batch index of each row (read only when mask != NULL)
 * query : [nrows] query index of each row (read only when causal != 0)
 */
void ref_softmax_fw(double *y, const double *x, const double *mask,
                    const int64_t *batch, const int64_t *query,
                    int64_t nrows, int64_t Tk, int causal)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const double *xr = x + r * Tk;
        double *yr = y + r * Tk;
        const double *mr = mask ? mask + batch[r] * Tk : 0;

        double m = -INFINITY;
        for (int64_t j = 0; j < Tk; ++j) {
            double z;
            if (causal && j > query[r])
                z = -INFINITY;
            else
                z = xr[j] + (mr ? mr[j] : 0.0);
            yr[j] = z;
            if (z > m)
                m = z;
        }
        if (m == -INFINITY) {
            for (int64_t j = 0; j < Tk; ++j)
                yr[j] = 0.0;
            continue;
        }
        double s = 0.0;
        for (int64_t j = 0; j < Tk; ++j) {
            double e = exp(yr[j] - m);
            yr[j] = e;
            s += e;
        }
        for (int64_t j = 0; j < Tk; ++j)
            yr[j] = yr[j] / s;
    }
}

/* ------------------------------------------------------------------------ */
/* Attention softmax backward                                                */
/* ------------------------------------------------------------------------ */
/*
 * Vector-Jacobian product of y = softmax(z) for each row:
 *   dx_j = y_j * (dy_j - sum_k y_k dy_k)
 * (the derivative dy_k/dz_j = y_k (delta_kj - y_j) contracted with dy).
 * Masked and future keys need no special case: their y is exactly 0.
 * dx, dy, y : [nrows, Tk]
 */
void ref_softmax_bw(double *dx, const double *dy, const double *y,
                    int64_t nrows, int64_t Tk)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const double *yr = y + r * Tk;
        const double *dyr = dy + r * Tk;
        double *dxr = dx + r * Tk;
        double s = 0.0;
        for (int64_t k = 0; k < Tk; ++k)
            s += yr[k] * dyr[k];
        for (int64_t j = 0; j < Tk; ++j)
            dxr[j] = yr[j] * (dyr[j] - s);
    }
}

/* ------------------------------------------------------------------------ */
/* Attention softmax, causal with Tq <= Tk, and the masked backward           */
/* ------------------------------------------------------------------------ */
/*
 * Visibility of key j to a row: not masked (mask != -inf) and, when causal,
 * not in the future.  With Tq queries over Tk >= Tq keys the queries are the
 * LAST Tq positions of the key sequence (bottom-right alignment): query i
 * sits at key position i + (Tk - Tq) and sees keys j <= i + (Tk - Tq).  For
 * Tq == Tk this is the j <= i rule of ref_softmax_fw.
 */
static int visible(const double *mr, int64_t j, int64_t q, int64_t offset, int causal)
{
    if (causal && j > q + offset)
        return 0;
    if (mr && mr[j] == -INFINITY)
        return 0;
    return 1;
}

/*
 * Softmax forward with a causal offset: as ref_softmax_fw, with future keys
 * j > query[r] + offset.  offset = Tk - Tq.
 */
void ref_softmax_fw_offset(double *y, const double *x, const double *mask,
                           const int64_t *batch, const int64_t *query,
                           int64_t nrows, int64_t Tk, int causal,
                           int64_t offset)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const double *xr = x + r * Tk;
        double *yr = y + r * Tk;
        const double *mr = mask ? mask + batch[r] * Tk : 0;
        const int64_t q = causal ? query[r] : 0;
        double m = -INFINITY;
        for (int64_t j = 0; j < Tk; ++j) {
            double z;
            if (causal && j > q + offset)
                z = -INFINITY;
            else
                z = xr[j] + (mr ? mr[j] : 0.0);
            yr[j] = z;
            if (z > m)
                m = z;
        }
        if (m == -INFINITY) {
            for (int64_t j = 0; j < Tk; ++j)
                yr[j] = 0.0;
            continue;
        }
        double s = 0.0;
        for (int64_t j = 0; j < Tk; ++j) {
            double e = exp(yr[j] - m);
            yr[j] = e;
            s += e;
        }
        for (int64_t j = 0; j < Tk; ++j)
            yr[j] = yr[j] / s;
    }
}

/*
 * Softmax backward restricted to the visible keys:
 *   s    = sum over visible k of y_k dy_k
 *   dx_j = y_j (dy_j - s)   for visible j,   0 otherwise.
 * When y is the forward output (exactly 0 on invisible keys) this equals
 * ref_softmax_bw; the masked form lets a kernel skip reading y and dy on keys
 * it knows are invisible.
 */
void ref_softmax_bw_masked(double *dx, const double *dy, const double *y,
                           const double *mask, const int64_t *batch,
                           const int64_t *query, int64_t nrows, int64_t Tk,
                           int causal, int64_t offset)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const double *yr = y + r * Tk;
        const double *dyr = dy + r * Tk;
        double *dxr = dx + r * Tk;
        const double *mr = mask ? mask + batch[r] * Tk : 0;
        const int64_t q = causal ? query[r] : 0;
        double s = 0.0;
        for (int64_t k = 0; k < Tk; ++k)
            if (visible(mr, k, q, offset, causal))
                s += yr[k] * dyr[k];
        for (int64_t j = 0; j < Tk; ++j)
            dxr[j] = visible(mr, j, q, offset, causal) ? yr[j] * (dyr[j] - s) : 0.0;
    }
}

/*
 * Scaled softmax forward (the fused "scale + mask + softmax" of an attention
 * layer): the scores are multiplied by `scale` (e.g. 1/sqrt(d)) before the
 * additive mask:
 *   z_j = -inf                          if causal and j > query[r] + offset
 *   z_j = scale * x_j + mask[b, j]      otherwise
 *   y   = exp(z - max z) / sum exp(z - max z)   (zeros when max z = -inf)
 */
void ref_softmax_fw_scaled(double *y, const double *x, const double *mask,
                           const int64_t *batch, const int64_t *query,
                           int64_t nrows, int64_t Tk, int causal,
                           int64_t offset, double scale)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const double *xr = x + r * Tk;
        double *yr = y + r * Tk;
        const double *mr = mask ? mask + batch[r] * Tk : 0;
        const int64_t q = causal ? query[r] : 0;
        double m = -INFINITY;
        for (int64_t j = 0; j < Tk; ++j) {
            double z = -INFINITY;
            if (!(causal && j > q + offset))
                z = scale * xr[j] + (mr ? mr[j] : 0.0);
            yr[j] = z;
            if (z > m)
                m = z;
        }
        if (m == -INFINITY) {
            for (int64_t j = 0; j < Tk; ++j)
                yr[j] = 0.0;
            continue;
        }
        double s = 0.0;
        for (int64_t j = 0; j < Tk; ++j) {
            yr[j] = exp(yr[j] - m);
            s += yr[j];
        }
        for (int64_t j = 0; j < Tk; ++j)
            yr[j] /= s;
    }
}

/*
 * Backward of the scaled softmax over the visible keys: with y the forward
 * output, d z_j / d x_j = scale, so
 *   s    = sum over visible k of y_k dy_k
 *   dx_j = scale * y_j * (dy_j - s)   for visible j,   0 otherwise.
 */
void ref_softmax_bw_masked_scaled(double *dx, const double *dy, const double *y,
                                  const double *mask, const int64_t *batch,
                                  const int64_t *query, int64_t nrows, int64_t Tk,
                                  int causal, int64_t offset, double scale)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const double *yr = y + r * Tk;
        const double *dyr = dy + r * Tk;
        double *dxr = dx + r * Tk;
        const double *mr = mask ? mask + batch[r] * Tk : 0;
        const int64_t q = causal ? query[r] : 0;
        double s = 0.0;
        for (int64_t k = 0; k < Tk; ++k)
            if (visible(mr, k, q, offset, causal))
                s += yr[k] * dyr[k];
        for (int64_t j = 0; j < Tk; ++j)
            dxr[j] = visible(mr, j, q, offset, causal) ? scale * yr[j] * (dyr[j] - s) : 0.0;
    }
}

/* ------------------------------------------------------------------------ */
/* LayerNorm forward                                                         */
/* ------------------------------------------------------------------------ */
/*
 * Two-pass textbook definition, per row of x [rows, N]:
 *   mu   = (1/N) sum_j x_j
 *   var  = (1/N) sum_j (x_j - mu)^2          (population variance)
 *   rstd = 1 / sqrt(var + eps)               (eps inside the root, [HW4] 2.1)
 *   y_j  = (x_j - mu) * rstd * gamma_j + beta_j
 * The kernels reach the same numbers with the one-pass rewrite of [L10]
 * slide 21; that rewrite is NOT used here.
 * y, x : [rows, N];  gamma, beta : [N];  mean, rstd : [rows]
 */
void ref_layernorm_fw(double *y, double *mean, double *rstd, const double *x,
                      const double *gamma, const double *beta,
                      int64_t rows, int64_t N, double eps)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * N;
        double *yr = y + r * N;
        double mu = 0.0;
        for (int64_t j = 0; j < N; ++j)
            mu += xr[j];
        mu /= (double)N;
        double var = 0.0;
        for (int64_t j = 0; j < N; ++j)
            var += (xr[j] - mu) * (xr[j] - mu);
        var /= (double)N;
        double rs = 1.0 / sqrt(var + eps);
        for (int64_t j = 0; j < N; ++j)
            yr[j] = (xr[j] - mu) * rs * gamma[j] + beta[j];
        mean[r] = mu;
        rstd[r] = rs;
    }
}

/*
 * The one-pass variance of [L10] slide 21, mu(x^2) - mu(x)^2, evaluated in
 * double (single == 0) or with float accumulation (single != 0).  Used only by
 * the tests that compare it with the two-pass definition; no other oracle
 * function calls it.
 */
double ref_variance_one_pass(const double *x, int64_t N, int single)
{
    if (single) {
        float s1 = 0.0f, s2 = 0.0f;
        for (int64_t j = 0; j < N; ++j) {
            float v = (float)x[j];
            s1 += v;
            s2 += v * v;
        }
        float m1 = s1 / (float)N, m2 = s2 / (float)N;
        return (double)(m2 - m1 * m1);
    }
    double s1 = 0.0, s2 = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        s1 += x[j];
        s2 += x[j] * x[j];
    }
    double m1 = s1 / (double)N, m2 = s2 / (double)N;
    return m2 - m1 * m1;
}

/* Two-pass population variance of one row (for the same comparison). */
double ref_variance_two_pass(const double *x, int64_t N)
{
    double mu = 0.0;
    for (int64_t j = 0; j < N; ++j)
        mu += x[j];
    mu /= (double)N;
    double var = 0.0;
    for (int64_t j = 0; j < N; ++j)
        var += (x[j] - mu) * (x[j] - mu);
    return var / (double)N;
}

/* ------------------------------------------------------------------------ */
/* LayerNorm backward: input gradient                                        */
/* ------------------------------------------------------------------------ */
/*
 * Closed-form gradient of y = (x - mu) * rstd * gamma + beta with respect to
 * x, where mu and rstd are the row statistics (given, as saved by the
 * forward pass):
 *   xhat_j = (x_j - mu) * rstd
 *   g_j    = gamma_j * dy_j
 *   dx_j   = rstd * ( g_j - (1/N) sum_k g_k - xhat_j * (1/N) sum_k g_k xhat_k )
 * The two sums are the ones [L10] slide 22 says can run in parallel.
 * dx, dy, x : [rows, N];  gamma : [N];  mean, rstd : [rows]
 */
void ref_layernorm_bw_dinp(double *dx, const double *dy, const double *x,
                           const double *gamma, const double *mean,
                           const double *rstd, int64_t rows, int64_t N)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * N;
        const double *dyr = dy + r * N;
        double *dxr = dx + r * N;
        double sum_g = 0.0, sum_gx = 0.0;
        for (int64_t k = 0; k < N; ++k) {
            double xhat = (xr[k] - mean[r]) * rstd[r];
            double g = gamma[k] * dyr[k];
            sum_g += g;
            sum_gx += g * xhat;
        }
        double a = sum_g / (double)N, b = sum_gx / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double xhat = (xr[j] - mean[r]) * rstd[r];
            double g = gamma[j] * dyr[j];
            dxr[j] = rstd[r] * (g - a - xhat * b);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* LayerNorm backward: gamma / beta gradients                                */
/* ------------------------------------------------------------------------ */
/*
 * Column sums over all rows ([HW4] Problem 2.2, the cross-row kernel):
 *   dgamma_j = sum_r dy_rj * (x_rj - mean_r) * rstd_r
 *   dbeta_j  = sum_r dy_rj
 * summed in row order.
 * dy, x : [rows, N];  mean, rstd : [rows];  dgamma, dbeta : [N]
 */
void ref_layernorm_bw_dgamma_dbeta(double *dgamma, double *dbeta,
                                   const double *dy, const double *x,
                                   const double *mean, const double *rstd,
                                   int64_t rows, int64_t N)
{
    for (int64_t j = 0; j < N; ++j) {
        double dg = 0.0, db = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
            double xhat = (x[r * N + j] - mean[r]) * rstd[r];
            dg += dy[r * N + j] * xhat;
            db += dy[r * N + j];
        }
        dgamma[j] = dg;
        dbeta[j] = db;
    }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm ([FT] section 5.4)                                                */
/* ------------------------------------------------------------------------ */
/*
 * Per row of x [rows, N]:
 *   ms   = (1/N) sum_j x_j^2
 *   rstd = 1 / sqrt(ms + eps)
 *   y_j  = x_j * rstd * gamma_j
 * y, x : [rows, N];  gamma : [N];  rstd : [rows]
 */
void ref_rmsnorm_fw(double *y, double *rstd, const double *x, const double *gamma,
                    int64_t rows, int64_t N, double eps)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * N;
        double *yr = y + r * N;
        double ms = 0.0;
        for (int64_t j = 0; j < N; ++j)
            ms += xr[j] * xr[j];
        ms /= (double)N;
        double rs = 1.0 / sqrt(ms + eps);
        for (int64_t j = 0; j < N; ++j)
            yr[j] = xr[j] * rs * gamma[j];
        rstd[r] = rs;
    }
}

/*
 * Input gradient of y = x * rstd * gamma, rstd = (mean(x^2) + eps)^(-1/2),
 * given the saved rstd:
 *   xhat_j = x_j * rstd,   g_j = gamma_j * dy_j
 *   dx_j   = rstd * ( g_j - xhat_j * (1/N) sum_k g_k xhat_k )
 * (d rstd / d x_j = -rstd^3 x_j / N; the single sum is the RMSNorm analogue
 * of the two LayerNorm sums.)
 */
void ref_rmsnorm_bw_dinp(double *dx, const double *dy, const double *x,
                         const double *gamma, const double *rstd, int64_t rows, int64_t N)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * N;
        const double *dyr = dy + r * N;
        double *dxr = dx + r * N;
        double sum_gx = 0.0;
        for (int64_t k = 0; k < N; ++k)
            sum_gx += gamma[k] * dyr[k] * (xr[k] * rstd[r]);
        double b = sum_gx / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double xhat = xr[j] * rstd[r];
            double g = gamma[j] * dyr[j];
            dxr[j] = rstd[r] * (g - xhat * b);
        }
    }
}

/* dgamma_j = sum_r dy_rj * x_rj * rstd_r  (column sums in row order). */
void ref_rmsnorm_bw_dgamma(double *dgamma, const double *dy, const double *x,
                           const double *rstd, int64_t rows, int64_t N)
{
    for (int64_t j = 0; j < N; ++j) {
        double dg = 0.0;
        for (int64_t r = 0; r < rows; ++r)
            dg += dy[r * N + j] * (x[r * N + j] * rstd[r]);
        dgamma[j] = dg;
    }
}

/* ------------------------------------------------------------------------ */
/* Cross entropy over a vocabulary                            [L10-T1]      */
/* ------------------------------------------------------------------------ */
/*
 * For each row r of logits z [rows, V] with target class t = target[r]:
 *   m      = max_j z_j
 *   lse_r  = m + log( sum_j exp(z_j - m) )     (log of the softmax denominator)
 *   loss_r = lse_r - z_t                       (= -log softmax(z)_t)
 * t < 0  : ignored row, loss_r = lse_r = 0 (the row is not read).
 * t >= V : loss_r = lse_r = NaN.
 */
void ref_cross_entropy_fw(double *loss, double *lse, const double *z, const int32_t *target,
                          int64_t rows, int64_t V)
{
    for (int64_t r = 0; r < rows; ++r) {
        const int32_t t = target[r];
        if (t < 0) {
            loss[r] = 0.0;
            lse[r] = 0.0;
            continue;
        }
        if ((int64_t)t >= V) {
            loss[r] = NAN;
            lse[r] = NAN;
            continue;
        }
        const double *zr = z + r * V;
        double m = -INFINITY;
        for (int64_t j = 0; j < V; ++j)
            if (zr[j] > m) m = zr[j];
        double s = 0.0;
        for (int64_t j = 0; j < V; ++j)
            s += exp(zr[j] - m);
        lse[r] = m + log(s);
        loss[r] = lse[r] - zr[t];
    }
}

/*
 * Gradient of loss_r with respect to the logits, scaled by the upstream
 * gradient dloss_r of that row:
 *   dz_j = dloss_r * ( exp(z_j - lse_r) - [j == t] )
 * (softmax minus the one-hot target).  Ignored rows (t < 0) get 0; t >= V
 * gets NaN.
 */
void ref_cross_entropy_bw(double *dz, const double *z, const int32_t *target,
                          const double *lse, const double *dloss, int64_t rows, int64_t V)
{
    for (int64_t r = 0; r < rows; ++r) {
        const int32_t t = target[r];
        double *dzr = dz + r * V;
        const double *zr = z + r * V;
        for (int64_t j = 0; j < V; ++j) {
            if (t < 0)
                dzr[j] = 0.0;
            else if ((int64_t)t >= V)
                dzr[j] = NAN;
            else
                dzr[j] = dloss[r] * (exp(zr[j] - lse[r]) - (j == t ? 1.0 : 0.0));
        }
    }
}
