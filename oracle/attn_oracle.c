/*
 * attn_oracle.c -- float64 CPU oracle for exact attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (page "Hardware Acceleration & Custom Kernels",
 * section 2 "FlashAttention: SRAM Tiling & Online Softmax", the attention
 * formula):  O = softmax(scale * Q K^T) V, row by row, plus the per-row
 * log-sum-exp of the scaled logits.  The plain formula is written out with
 * no tiling: for each (batch, head, query row i)
 *
 *     s_j  = scale * sum_c q[i,c] k[j,c]        j in J_i
 *     m    = max_j s_j
 *     w_j  = exp(s_j - m)
 *     l    = sum_j w_j
 *     O[i] = sum_j w_j v[j] / l
 *     LSE  = m + ln l
 *
 * J_i = [0, N) without a mask; J_i = [0, i] with the causal mask (key j is
 * visible to query i iff j <= i).  The pages do not define the causal mask or
 * the LSE; those are the plainest readings and are listed with the design
 * notes.
 *
 * A second routine replays the same rows with the online-normalisation
 * recurrence of the same section (m_new = max(m_old, x),
 * d_new = d_old e^(m_old - m_new) + e^(x - m_new)), applied one key tile at
 * a time, with the output sums rescaled by the same factor.  It exists so the
 * tests can check that the tile-by-tile replay equals the one-shot formula
 * (the two-tile simulation that page's section 5 announces).
 *
 * Inputs are float32 arrays holding exactly the values the GPU sees (bf16
 * inputs are widened to float32 without rounding by the caller); every
 * product and sum is taken in double.  Layout: [B, H, N, d], d contiguous.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Scores of one query row against keys [0, nvis); returns their maximum. */
static double row_scores(const float *qrow, const float *K, int64_t nvis,
                         int64_t d, double scale, double *s)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        const float *krow = K + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += (double)qrow[c] * (double)krow[c];
        s[j] = scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    return m;
}

/* One query row of one (batch, head) slice, by the plain formula. */
static void one_row(const float *Q, const float *K, const float *V,
                    int64_t N, int64_t d, int64_t i, double scale, int causal,
                    double *s, double *orow, double *lse)
{
    const int64_t nvis = causal ? i + 1 : N;
    const double m = row_scores(Q + i * d, K, nvis, d, scale, s);
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            acc += s[j] * (double)V[j * d + c];
        orow[c] = acc / l;
    }
    *lse = m + log(l);
}

static int bad_shape(int64_t B, int64_t H, int64_t N, int64_t d)
{
    return B < 1 || H < 1 || N < 1 || d < 1;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Threads OpenMP will use for the next parallel region (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full forward: o [B,H,N,d] and lse [B,H,N] (lse may be NULL).
 * Returns 0, or -1 on a bad shape / allocation failure.
 */
int oracle_attn_fwd(const float *q, const float *k, const float *v,
                    double *o, double *lse,
                    int64_t B, int64_t H, int64_t N, int64_t d,
                    double scale, int causal, int nthreads)
{
    if (bad_shape(B, H, N, d) || !q || !k || !v || !o)
        return -1;
    set_threads(nthreads);
    const int64_t rows = B * H * N;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)N * sizeof(double));
        double lse_tmp;
        if (!s) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < rows; ++r) {
                const int64_t bh = r / N, i = r % N;
                const int64_t base = bh * N * d;
                one_row(q + base, k + base, v + base, N, d, i, scale, causal, s,
                        o + r * d, lse ? lse + r : &lse_tmp);
            }
            free(s);
        }
    }
    return failed ? -1 : 0;
}

/*
 * A chosen subset of rows: row t is query row rows[t] of slice bh[t]
 * (bh = b*H + h).  o is [nrows, d], lse [nrows].  Used to check sampled
 * outputs of workloads too large for the full oracle.
 */
int oracle_attn_fwd_rows(const float *q, const float *k, const float *v,
                         int64_t B, int64_t H, int64_t N, int64_t d,
                         double scale, int causal,
                         const int64_t *bh, const int64_t *rows, int64_t nrows,
                         double *o, double *lse, int nthreads)
{
    if (bad_shape(B, H, N, d) || !q || !k || !v || !o || !lse || nrows < 0)
        return -1;
    for (int64_t t = 0; t < nrows; ++t)
        if (bh[t] < 0 || bh[t] >= B * H || rows[t] < 0 || rows[t] >= N)
            return -1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)N * sizeof(double));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < nrows; ++t) {
                const int64_t base = bh[t] * N * d;
                one_row(q + base, k + base, v + base, N, d, rows[t], scale,
                        causal, s, o + t * d, lse + t);
            }
            free(s);
        }
    }
    return failed ? -1 : 0;
}

/*
 * The probability row P[i, :] = softmax_j(s_ij) of one (batch, head) slice
 * (q, k point at that slice).  Masked keys get probability 0.  p is [N].
 */
int oracle_probs_row(const float *q, const float *k, int64_t N, int64_t d,
                     int64_t i, double scale, int causal, double *p)
{
    if (N < 1 || d < 1 || i < 0 || i >= N || !p)
        return -1;
    const int64_t nvis = causal ? i + 1 : N;
    const double m = row_scores(q + i * d, k, nvis, d, scale, p);
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int64_t j = 0; j < nvis; ++j)
        p[j] /= l;
    for (int64_t j = nvis; j < N; ++j)
        p[j] = 0.0;
    return 0;
}

/*
 * Online replay over one (batch, head) slice: keys are visited in tiles of
 * `tile` keys.  Per query row the running maximum m, running normaliser l and
 * running output sum acc are updated per tile as
 *     m'   = max(m, max over the tile of s_j)
 *     l'   = l e^(m - m') + sum over the tile of e^(s_j - m')
 *     acc' = acc e^(m - m') + sum over the tile of e^(s_j - m') v_j
 * and O = acc / l, LSE = m + ln l at the end.  o is [N, d], lse [N].
 */
int oracle_online_replay(const float *q, const float *k, const float *v,
                         int64_t N, int64_t d, double scale, int causal,
                         int64_t tile, double *o, double *lse)
{
    if (N < 1 || d < 1 || tile < 1 || !o || !lse)
        return -1;
    double *s = (double *)malloc((size_t)tile * sizeof(double));
    double *acc = (double *)malloc((size_t)d * sizeof(double));
    if (!s || !acc) {
        free(s);
        free(acc);
        return -1;
    }
    for (int64_t i = 0; i < N; ++i) {
        const int64_t nvis = causal ? i + 1 : N;
        double m = -INFINITY, l = 0.0;
        memset(acc, 0, (size_t)d * sizeof(double));
        for (int64_t j0 = 0; j0 < nvis; j0 += tile) {
            const int64_t nt = (nvis - j0 < tile) ? nvis - j0 : tile;
            const double tmax = row_scores(q + i * d, k + j0 * d, nt, d, scale, s);
            const double m_new = (tmax > m) ? tmax : m;
            const double alpha = exp(m - m_new); /* exp(-inf) = 0 on the first tile */
            l *= alpha;
            for (int64_t c = 0; c < d; ++c)
                acc[c] *= alpha;
            for (int64_t j = 0; j < nt; ++j) {
                const double w = exp(s[j] - m_new);
                l += w;
                for (int64_t c = 0; c < d; ++c)
                    acc[c] += w * (double)v[(j0 + j) * d + c];
            }
            m = m_new;
        }
        for (int64_t c = 0; c < d; ++c)
            o[i * d + c] = acc[c] / l;
        lse[i] = m + log(l);
    }
    free(s);
    free(acc);
    return 0;
}

/*
 * Row softmax of a [rows, width] matrix (page "14. Triton and kernel fusion",
 * section "Fusion": subtract the row maximum, exponentiate, divide by the
 * row sum).  y is [rows, width], lse [rows] (may be NULL) = max + ln(sum).
 */
int oracle_row_softmax(const float *x, int64_t rows, int64_t width,
                       double *y, double *lse, int nthreads)
{
    if (rows < 1 || width < 1 || !x || !y)
        return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * width;
        double *yr = y + r * width;
        double m = -INFINITY;
        for (int64_t c = 0; c < width; ++c)
            if ((double)xr[c] > m)
                m = (double)xr[c];
        double l = 0.0;
        for (int64_t c = 0; c < width; ++c) {
            yr[c] = exp((double)xr[c] - m);
            l += yr[c];
        }
        for (int64_t c = 0; c < width; ++c)
            yr[c] /= l;
        if (lse)
            lse[r] = m + log(l);
    }
    return 0;
}

/*
 * Residual add + RMSNorm of a [rows, width] matrix (page "14. Triton and
 * kernel fusion", section "Fused residual add + RMSNorm"; the normalisation
 * of page "TritonForge": x / sqrt(sum x_i^2 / d + eps) * gamma):
 *     h   = x + residual           (h = x when residual is NULL)
 *     out = h / sqrt(mean_c h_c^2 + eps) * weight
 * h_out (may be NULL) receives h.  All in double.
 */
int oracle_add_rmsnorm(const float *x, const float *residual, const float *weight,
                       int64_t rows, int64_t width, double eps, double *out, double *h_out,
                       int nthreads)
{
    if (rows < 1 || width < 1 || !x || !weight || !out)
        return -1;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *h = (double *)malloc((size_t)width * sizeof(double));
        if (h) {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < rows; ++r) {
                double ss = 0.0;
                for (int64_t c = 0; c < width; ++c) {
                    h[c] = (double)x[r * width + c] +
                           (residual ? (double)residual[r * width + c] : 0.0);
                    ss += h[c] * h[c];
                }
                const double inv = 1.0 / sqrt(ss / (double)width + eps);
                for (int64_t c = 0; c < width; ++c) {
                    out[r * width + c] = h[c] * inv * (double)weight[c];
                    if (h_out)
                        h_out[r * width + c] = h[c];
                }
            }
            free(h);
        }
    }
    return 0;
}

/*
 * Attention backward over one (batch, head) slice, the exact gradient of the
 * forward formula given the forward's outputs O and LSE:
 *     P_ij  = exp(scale q_i.k_j - LSE_i)        (0 for masked keys)
 *     D_i   = sum_c dO_ic O_ic
 *     dP_ij = dO_i . v_j
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale sum_j dS_ij k_j
 *     dK_j  = scale sum_i dS_ij q_i
 *     dV_j  = sum_i P_ij dO_i
 * The pages give no attention backward; this is the plain derivative.  All
 * arrays are one slice, [N, d] (lse [N]); outputs are double.
 */
static int bwd_slice(const float *q, const float *k, const float *v, const float *o,
                     const float *dout, const float *lse, int64_t N, int64_t d, double scale,
                     int causal, double *dq, double *dk, double *dv)
{
    memset(dk, 0, (size_t)(N * d) * sizeof(double));
    memset(dv, 0, (size_t)(N * d) * sizeof(double));
    for (int64_t i = 0; i < N; ++i) {
        const int64_t nvis = causal ? i + 1 : N;
        double Di = 0.0;
        for (int64_t c = 0; c < d; ++c)
            Di += (double)dout[i * d + c] * (double)o[i * d + c];
        for (int64_t c = 0; c < d; ++c)
            dq[i * d + c] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            double s = 0.0, dp = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                s += (double)q[i * d + c] * (double)k[j * d + c];
                dp += (double)dout[i * d + c] * (double)v[j * d + c];
            }
            const double pij = exp(scale * s - (double)lse[i]);
            const double ds = pij * (dp - Di);
            for (int64_t c = 0; c < d; ++c) {
                dq[i * d + c] += scale * ds * (double)k[j * d + c];
                dk[j * d + c] += scale * ds * (double)q[i * d + c];
                dv[j * d + c] += pij * (double)dout[i * d + c];
            }
        }
    }
    return 0;
}

/* Backward for all slices of [B, H, N, d] tensors (OpenMP over slices). */
int oracle_attn_bwd(const float *q, const float *k, const float *v, const float *o,
                    const float *dout, const float *lse, int64_t B, int64_t H, int64_t N,
                    int64_t d, double scale, int causal, double *dq, double *dk, double *dv,
                    int nthreads)
{
    if (bad_shape(B, H, N, d) || !q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
        return -1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const int64_t base = bh * N * d;
        if (bwd_slice(q + base, k + base, v + base, o + base, dout + base, lse + bh * N, N, d,
                      scale, causal, dq + base, dk + base, dv + base) != 0) {
#pragma omp atomic write
            failed = 1;
        }
    }
    return failed ? -1 : 0;
}
