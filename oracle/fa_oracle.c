/*
 * fa_oracle.c -- plain, slow, float64 CPU oracle for exact scaled-dot-product
 * attention and its gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA path, and the CUDA path never calls
 * it.
 *
 * What it computes (the plain definition, not the tiled algorithm):
 *   "Learning Metal with FlashAttention", section "FlashAttention": for each
 *   query row i, o_i = sum_j softmax_j(s_ij) v_j over the whole score row
 *   s_i:, made numerically stable by subtracting the row maximum first.
 *   "Flash Attention" (metalworking), kernel anatomy item 4: the causal case
 *   is key j visible to query i iff j <= i (self-attention, N_q = N_k).
 *   "FlashAttention (Metal port)" (metal-flash-attention), section on
 *   quantifying performance, forward pseudocode: L = m + log_e(l), the
 *   natural log-sum-exp of the scaled scores.
 *   Same page, backward pseudocode: D_i = rowsum(dO_i * O_i), P = exp(S - L),
 *   dP = dO V^T, dS = P * (dP - D) * scale, dQ = dS K, dK = dS^T Q,
 *   dV = P^T dO.  (The page prints "D = dO * O"; the only shape-consistent
 *   reading is the row sum, which is also the chain rule for softmax.)
 *
 * Every score row is materialised in full: there is no online softmax, no
 * tiling and no reordering.  Exponentials are natural (exp in double); the
 * base-2 form is a kernel implementation choice and does not appear here.
 *
 * One call handles one (batch, head) slice: q, k, v, dO are [N, D] row-major
 * float64.  Callers loop over heads (and may run heads on several threads).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Number of keys query row i may attend to: all N, or 0..i when causal. */
static int64_t visible_keys(int64_t i, int64_t N, int causal)
{
    return causal ? i + 1 : N;
}

/* s_j = scale * <q_i, k_j> for j < nvis. */
static void score_row(const double *q_i, const double *k, int64_t nvis, int64_t D,
                      double scale, double *s)
{
    for (int64_t j = 0; j < nvis; ++j) {
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d)
            acc += q_i[d] * k[j * D + d];
        s[j] = scale * acc;
    }
}

/* In place: s_j <- exp(s_j - m) / l with m = max_j s_j, l = sum_j exp(s_j - m).
 * Returns the natural log-sum-exp m + ln(l). */
static double softmax_row(double *s, int64_t n)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (s[j] > m)
            m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t j = 0; j < n; ++j)
        s[j] /= l;
    return m + log(l);
}

/*
 * Forward for selected query rows of one head.
 *   rows   : n_rows query indices (NULL means rows 0..n_rows-1)
 *   o      : [n_rows, D] output
 *   lse    : [n_rows]    natural log-sum-exp of the scaled scores
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int fa_oracle_forward_rows(const double *q, const double *k, const double *v,
                           int64_t N, int64_t D, double scale, int causal,
                           int64_t n_rows, const int64_t *rows,
                           double *o, double *lse)
{
    if (N < 1 || D < 1 || n_rows < 0)
        return -1;
    double *p = (double *)malloc((size_t)N * sizeof(double));
    if (!p)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= N) {
            free(p);
            return -1;
        }
        int64_t nvis = visible_keys(i, N, causal);
        score_row(q + i * D, k, nvis, D, scale, p);
        lse[r] = softmax_row(p, nvis);
        /* O_i = sum_j P_ij v_j */
        for (int64_t d = 0; d < D; ++d)
            o[r * D + d] = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            for (int64_t d = 0; d < D; ++d)
                o[r * D + d] += p[j] * v[j * D + d];
    }
    free(p);
    return 0;
}

/*
 * Forward + backward contributions of query rows [row_begin, row_end) of one
 * head, the plain definition row by row.  For each such row i it writes
 * o[i], lse[i], delta[i], dq[i] and ADDS row i's terms to dk and dv (the
 * caller zeroes them; over all rows 0..N-1 they become the full gradients).
 *   o, lse        : [N, D], [N]      forward outputs (float64, exact up to rounding)
 *   delta         : [N]              D_i = sum_d dO_id * O_id (this oracle's own O)
 *   dq, dk, dv    : [N, D]           gradients of sum(O * dO)
 * o, lse and delta may be NULL.
 */
int fa_oracle_backward_head_rows(const double *q, const double *k, const double *v,
                                 const double *dO, int64_t N, int64_t D, double scale,
                                 int causal, int64_t row_begin, int64_t row_end,
                                 double *o, double *lse, double *delta,
                                 double *dq, double *dk, double *dv)
{
    if (N < 1 || D < 1 || !dq || !dk || !dv || row_begin < 0 || row_end > N ||
        row_begin > row_end)
        return -1;
    double *p = (double *)malloc((size_t)N * sizeof(double));
    double *orow = (double *)malloc((size_t)D * sizeof(double));
    if (!p || !orow) {
        free(p);
        free(orow);
        return -1;
    }
    for (int64_t i = row_begin; i < row_end; ++i) {
        int64_t nvis = visible_keys(i, N, causal);
        const double *q_i = q + i * D;
        const double *do_i = dO + i * D;
        /* P_i: = softmax of the scaled score row */
        score_row(q_i, k, nvis, D, scale, p);
        double lse_i = softmax_row(p, nvis);
        /* O_i = sum_j P_ij v_j */
        for (int64_t d = 0; d < D; ++d)
            orow[d] = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            for (int64_t d = 0; d < D; ++d)
                orow[d] += p[j] * v[j * D + d];
        /* D_i = sum_d dO_id O_id */
        double delta_i = 0.0;
        for (int64_t d = 0; d < D; ++d)
            delta_i += do_i[d] * orow[d];
        if (o)
            memcpy(o + i * D, orow, (size_t)D * sizeof(double));
        if (lse)
            lse[i] = lse_i;
        if (delta)
            delta[i] = delta_i;
        for (int64_t d = 0; d < D; ++d)
            dq[i * D + d] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            /* dP_ij = <dO_i, v_j>; dS_ij = P_ij (dP_ij - D_i) scale */
            double dp = 0.0;
            for (int64_t d = 0; d < D; ++d)
                dp += do_i[d] * v[j * D + d];
            double ds = p[j] * (dp - delta_i) * scale;
            for (int64_t d = 0; d < D; ++d) {
                dq[i * D + d] += ds * k[j * D + d];   /* dQ = dS K    */
                dk[j * D + d] += ds * q_i[d];         /* dK = dS^T Q  */
                dv[j * D + d] += p[j] * do_i[d];      /* dV = P^T dO  */
            }
        }
    }
    free(p);
    free(orow);
    return 0;
}

/* Full forward + backward of one head: all rows of fa_oracle_backward_head_rows. */
int fa_oracle_backward_head(const double *q, const double *k, const double *v,
                            const double *dO, int64_t N, int64_t D, double scale,
                            int causal, double *o, double *lse, double *delta,
                            double *dq, double *dk, double *dv)
{
    if (N < 1 || D < 1 || !dq || !dk || !dv)
        return -1;
    memset(dk, 0, (size_t)(N * D) * sizeof(double));
    memset(dv, 0, (size_t)(N * D) * sizeof(double));
    return fa_oracle_backward_head_rows(q, k, v, dO, N, D, scale, causal, 0, N, o, lse, delta,
                                        dq, dk, dv);
}

/*
 * dQ and D for selected query rows of one head (each row needs only its own
 * score row and all of K, V).
 *   dq    : [n_rows, D],  delta : [n_rows]
 */
int fa_oracle_backward_dq_rows(const double *q, const double *k, const double *v,
                               const double *dO, int64_t N, int64_t D, double scale,
                               int causal, int64_t n_rows, const int64_t *rows,
                               double *dq, double *delta)
{
    if (N < 1 || D < 1 || n_rows < 0)
        return -1;
    double *p = (double *)malloc((size_t)N * sizeof(double));
    double *orow = (double *)malloc((size_t)D * sizeof(double));
    if (!p || !orow) {
        free(p);
        free(orow);
        return -1;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= N) {
            free(p);
            free(orow);
            return -1;
        }
        int64_t nvis = visible_keys(i, N, causal);
        const double *do_i = dO + i * D;
        score_row(q + i * D, k, nvis, D, scale, p);
        softmax_row(p, nvis);
        for (int64_t d = 0; d < D; ++d)
            orow[d] = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            for (int64_t d = 0; d < D; ++d)
                orow[d] += p[j] * v[j * D + d];
        double delta_i = 0.0;
        for (int64_t d = 0; d < D; ++d)
            delta_i += do_i[d] * orow[d];
        if (delta)
            delta[r] = delta_i;
        for (int64_t d = 0; d < D; ++d)
            dq[r * D + d] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            double dp = 0.0;
            for (int64_t d = 0; d < D; ++d)
                dp += do_i[d] * v[j * D + d];
            double ds = p[j] * (dp - delta_i) * scale;
            for (int64_t d = 0; d < D; ++d)
                dq[r * D + d] += ds * k[j * D + d];
        }
    }
    free(p);
    free(orow);
    return 0;
}

/*
 * dK and dV for selected key rows of one head.  Column j of P needs the
 * normaliser of every query row that sees key j, so the caller passes the
 * natural log-sum-exp lse[i] and D_i = delta[i] of ALL N query rows (from
 * fa_oracle_forward_rows / fa_oracle_backward_dq_rows of this oracle); then
 * P_ij = exp(s_ij - lse_i), which is the softmax by definition of lse.
 *   dk, dv : [n_rows, D]
 */
int fa_oracle_backward_dkdv_rows(const double *q, const double *k, const double *v,
                                 const double *dO, const double *lse,
                                 const double *delta, int64_t N, int64_t D,
                                 double scale, int causal, int64_t n_rows,
                                 const int64_t *rows, double *dk, double *dv)
{
    if (N < 1 || D < 1 || n_rows < 0)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t j = rows ? rows[r] : r;
        if (j < 0 || j >= N)
            return -1;
        const double *k_j = k + j * D;
        const double *v_j = v + j * D;
        for (int64_t d = 0; d < D; ++d) {
            dk[r * D + d] = 0.0;
            dv[r * D + d] = 0.0;
        }
        for (int64_t i = causal ? j : 0; i < N; ++i) {
            const double *q_i = q + i * D;
            const double *do_i = dO + i * D;
            double s = 0.0, dp = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                s += q_i[d] * k_j[d];
                dp += do_i[d] * v_j[d];
            }
            double p = exp(scale * s - lse[i]);
            double ds = p * (dp - delta[i]) * scale;
            for (int64_t d = 0; d < D; ++d) {
                dk[r * D + d] += ds * q_i[d];
                dv[r * D + d] += p * do_i[d];
            }
        }
    }
    return 0;
}

/*
 * Decode form: n_q query rows against N_k keys of one head (q is [n_q, D],
 * k and v are [N_k, D]).  The query rows are the LAST n_q positions of the
 * sequence, so with causal masking query row i sees keys j <= N_k - n_q + i
 * (for n_q = N_k this is the self-attention rule above); without it every
 * row sees all N_k keys.  Same plain definition: full score row, row-max
 * shifted softmax, O_i = sum_j P_ij v_j, lse_i = m_i + ln(l_i).
 *   o : [n_q, D],  lse : [n_q]
 */
int fa_oracle_forward_kv(const double *q, const double *k, const double *v,
                         int64_t n_q, int64_t N_k, int64_t D, double scale, int causal,
                         double *o, double *lse)
{
    if (n_q < 1 || N_k < 1 || D < 1 || n_q > N_k)
        return -1;
    double *p = (double *)malloc((size_t)N_k * sizeof(double));
    if (!p)
        return -1;
    for (int64_t i = 0; i < n_q; ++i) {
        int64_t nvis = causal ? N_k - n_q + i + 1 : N_k;
        score_row(q + i * D, k, nvis, D, scale, p);
        lse[i] = softmax_row(p, nvis);
        for (int64_t d = 0; d < D; ++d)
            o[i * D + d] = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            for (int64_t d = 0; d < D; ++d)
                o[i * D + d] += p[j] * v[j * D + d];
    }
    free(p);
    return 0;
}
