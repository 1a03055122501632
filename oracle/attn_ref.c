/*
 * Oracle for softmax attention, fp64, plain C.  TEST INFRASTRUCTURE ONLY:
 * nothing in the product path may link, load or call this file.
 *
 * What it computes, per (batch b, head h), for query row i:
 *
 *     s_ij = scale * sum_c q_ic k_jc                       (score row, fully materialised)
 *     s_ij = -inf                      if causal and j > i (query i sees keys 0..i)
 *     m_i  = max_j s_ij
 *     e_ij = exp(s_ij - m_i),  l_i = sum_j e_ij,  P_ij = e_ij / l_i
 *     O_ic = sum_j P_ij v_jc
 *     L_i  = m_i + ln l_i                                   (logsumexp, natural log)
 *
 * Sources:
 *   - "Kernels — fusion and FlashAttention" (jiahuanglin.xyz cs336 lesson 07),
 *     §2 "Naive attention": scores, mask, softmax, weight the values; the
 *     tensors are (B, h, T, d_head).
 *   - same page, §3: softmax subtracts the row max for stability before
 *     exponentiating and divides by the row sum.
 *   - same page, §5: the forward saves m + log(l) per row (logsumexp).
 *   - "Writing and Benchmarking Custom Kernels" (arunshar.com, ch. 10),
 *     §10.3.1: S = QK^T / sqrt(d), m_i = max_j S_ij, denominator
 *     sum_j exp(S_ij - m_i); §10.3.2: L_i = m_i + log l_i kept in fp32 by
 *     the kernel (the oracle keeps fp64).
 *   - same chapter, §10.3.1 "What you actually decide": causal masking drops
 *     the key tiles above the diagonal.
 *
 * A second routine, oracle_attn_online_f64, carries out the tile-by-tile
 * online-softmax recurrence of "Kernels — fusion and FlashAttention" §3 (running
 * max m, running denominator l, running output o, each rescaled by
 * exp(m_old - m_new) when a tile raises the max; out = o / l), in fp64, so that
 * tests can check that the recurrence reaches the two-pass result.
 *
 * Inputs are bf16 bit patterns (uint16), widened exactly to fp64.  Layout is
 * contiguous (B, H, N, d) row-major for q, k, v and o; (B, H, N) for lse.
 * Nothing here is blocked, fused or reordered beyond the definition: the only
 * parallelism is independent query rows spread over OpenMP threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One query row i of one (b, h): materialise the score row, mask, two-pass
 * softmax, P.V and the logsumexp.  s_row is caller-provided scratch of N
 * doubles.  p_row (nullable) receives the probability row. */
static void attention_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t N, int64_t d, int causal, double scale, int64_t i,
                          double *s_row, double *o_row, double *lse, double *p_row)
{
    /* scores */
    for (int64_t j = 0; j < N; ++j) {
        if (causal && j > i) {
            s_row[j] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += bf16_bits_to_f64(q[i * d + c]) * bf16_bits_to_f64(k[j * d + c]);
        s_row[j] = scale * acc;
    }
    /* pass 1: row max */
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j)
        if (s_row[j] > m) m = s_row[j];
    /* pass 2: exponentials and their sum */
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        s_row[j] = exp(s_row[j] - m); /* exp(-inf) = 0 for masked keys */
        l += s_row[j];
    }
    /* normalise, then weight the values */
    for (int64_t j = 0; j < N; ++j) s_row[j] /= l;
    if (p_row)
        for (int64_t j = 0; j < N; ++j) p_row[j] = s_row[j];
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        const double p = s_row[j];
        if (p == 0.0) continue;
        for (int64_t c = 0; c < d; ++c) o_row[c] += p * bf16_bits_to_f64(v[j * d + c]);
    }
    *lse = m + log(l);
}

static int bad_shape(int64_t B, int64_t H, int64_t N, int64_t d)
{
    return B < 1 || H < 1 || N < 1 || d < 1;
}

static int pick_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Full tensor.  o: B*H*N*d doubles, lse: B*H*N doubles, p (nullable):
 * B*H*N*N doubles.  Returns 0 on success, -1 on bad arguments, -2 on
 * allocation failure. */
int oracle_attn_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                    double *o, double *lse, double *p, int nthreads)
{
    if (!q || !k || !v || !o || !lse || bad_shape(B, H, N, d)) return -1;
    const int64_t rows = B * H * N;
    int failed = 0;
#pragma omp parallel num_threads(pick_threads(nthreads))
    {
        double *s_row = (double *)malloc((size_t)N * sizeof(double));
        if (!s_row) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!s_row) continue;
            const int64_t bh = r / N, i = r % N;
            const int64_t head = bh * N * d;
            attention_row(q + head, k + head, v + head, N, d, causal, scale, i, s_row,
                          o + r * d, lse + r, p ? p + r * N : NULL);
        }
        free(s_row);
    }
    return failed ? -2 : 0;
}

/* Selected rows only: row t is query row_idx[t] of flattened head bh_idx[t]
 * (bh = b*H + h).  o_rows: nrows*d, lse_rows: nrows. */
int oracle_attn_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                         const int64_t *bh_idx, const int64_t *row_idx, int64_t nrows,
                         double *o_rows, double *lse_rows, int nthreads)
{
    if (!q || !k || !v || !bh_idx || !row_idx || !o_rows || !lse_rows || nrows < 0 ||
        bad_shape(B, H, N, d))
        return -1;
    for (int64_t t = 0; t < nrows; ++t)
        if (bh_idx[t] < 0 || bh_idx[t] >= B * H || row_idx[t] < 0 || row_idx[t] >= N) return -1;
    int failed = 0;
#pragma omp parallel num_threads(pick_threads(nthreads))
    {
        double *s_row = (double *)malloc((size_t)N * sizeof(double));
        if (!s_row) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < nrows; ++t) {
            if (!s_row) continue;
            const int64_t head = bh_idx[t] * N * d;
            attention_row(q + head, k + head, v + head, N, d, causal, scale, row_idx[t], s_row,
                          o_rows + t * d, lse_rows + t, NULL);
        }
        free(s_row);
    }
    return failed ? -2 : 0;
}

/* The online-softmax recurrence, keys taken `tile` at a time.  For each query
 * row: m = -inf, l = 0, o = 0; for each key tile: scores s of the tile (masked
 * keys at -inf), m_new = max(m, max s), c = exp(m - m_new),
 * p = exp(s - m_new), l = l*c + sum p, o = o*c + p.V_tile, m = m_new; finally
 * out = o / l and lse = m + ln l.  Under the causal mask a tile whose every
 * key lies above the diagonal is skipped (it adds nothing). */
int oracle_attn_online_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                           int64_t tile, double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || tile < 1 || bad_shape(B, H, N, d)) return -1;
    const int64_t rows = B * H * N;
    int failed = 0;
#pragma omp parallel num_threads(pick_threads(nthreads))
    {
        double *s = (double *)malloc((size_t)tile * sizeof(double));
        double *acc = (double *)malloc((size_t)d * sizeof(double));
        if (!s || !acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!s || !acc) continue;
            const int64_t bh = r / N, i = r % N;
            const uint16_t *qh = q + bh * N * d, *kh = k + bh * N * d, *vh = v + bh * N * d;
            double m = -INFINITY, l = 0.0;
            for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
            for (int64_t j0 = 0; j0 < N; j0 += tile) {
                if (causal && j0 > i) break; /* tile entirely above the diagonal */
                const int64_t n = (j0 + tile <= N) ? tile : N - j0;
                double tile_max = -INFINITY;
                for (int64_t t = 0; t < n; ++t) {
                    const int64_t j = j0 + t;
                    if (causal && j > i) {
                        s[t] = -INFINITY;
                        continue;
                    }
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c)
                        dot += bf16_bits_to_f64(qh[i * d + c]) * bf16_bits_to_f64(kh[j * d + c]);
                    s[t] = scale * dot;
                    if (s[t] > tile_max) tile_max = s[t];
                }
                const double m_new = (tile_max > m) ? tile_max : m;
                const double corr = exp(m - m_new); /* exp(-inf) = 0 on the first tile */
                double psum = 0.0;
                for (int64_t c = 0; c < d; ++c) acc[c] *= corr;
                for (int64_t t = 0; t < n; ++t) {
                    const double p = exp(s[t] - m_new);
                    psum += p;
                    if (p == 0.0) continue;
                    const int64_t j = j0 + t;
                    for (int64_t c = 0; c < d; ++c) acc[c] += p * bf16_bits_to_f64(vh[j * d + c]);
                }
                l = l * corr + psum;
                m = m_new;
            }
            for (int64_t c = 0; c < d; ++c) o[r * d + c] = acc[c] / l;
            lse[r] = m + log(l);
        }
        free(s);
        free(acc);
    }
    return failed ? -2 : 0;
}

/* ------------------------------------------------------------------------
 * Rectangular attention (decode): Nq query rows against a cache of Nk keys.
 * Query i stands at key position Nk - Nq + i (the newest Nq keys belong to
 * the queries), so under the causal mask it sees keys 0 .. Nk - Nq + i;
 * without the mask it sees all Nk.  For one query (the decode step of
 * "Fusion and IO-aware kernels", section "Where it breaks": one query token
 * per sequence, reading the whole KV cache) both are the same.  Each row is
 * the same definition as above: scores, mask, two-pass softmax, P.V,
 * logsumexp.  q, o: (B, H, Nq, d); k, v: (B, H, Nk, d); lse: (B, H, Nq).
 * ------------------------------------------------------------------------ */
static void attention_row_keys(const uint16_t *q_row, const uint16_t *k, const uint16_t *v,
                               int64_t Nk, int64_t d, int64_t last_key, double scale,
                               double *s_row, double *o_row, double *lse)
{
    for (int64_t j = 0; j < Nk; ++j) {
        if (j > last_key) {
            s_row[j] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += bf16_bits_to_f64(q_row[c]) * bf16_bits_to_f64(k[j * d + c]);
        s_row[j] = acc * scale;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < Nk; ++j)
        if (s_row[j] > m) m = s_row[j];
    double l = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        const double e = exp(s_row[j] - m);
        s_row[j] = e;
        l += e;
    }
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        const double pj = s_row[j] / l;
        if (pj == 0.0) continue;
        for (int64_t c = 0; c < d; ++c) o_row[c] += pj * bf16_bits_to_f64(v[j * d + c]);
    }
    *lse = log(l) + m;
}

static int bad_rect(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal)
{
    return B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || (causal && Nq > Nk);
}

/* Full tensor.  o: B*H*Nq*d doubles, lse: B*H*Nq doubles. */
int oracle_attn_rect_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                         int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal, double scale,
                         double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || bad_rect(B, H, Nq, Nk, d, causal)) return -1;
    const int64_t rows = B * H * Nq;
    int failed = 0;
#pragma omp parallel num_threads(pick_threads(nthreads))
    {
        double *s_row = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s_row) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < rows; ++r) {
            if (!s_row) continue;
            const int64_t bh = r / Nq, i = r % Nq;
            const int64_t last = causal ? Nk - Nq + i : Nk - 1;
            attention_row_keys(q + r * d, k + bh * Nk * d, v + bh * Nk * d, Nk, d, last, scale,
                               s_row, o + r * d, lse + r);
        }
        free(s_row);
    }
    return failed ? -2 : 0;
}

/* Selected rows: row t is query row_idx[t] of flattened head bh_idx[t]. */
int oracle_attn_rect_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal,
                              double scale, const int64_t *bh_idx, const int64_t *row_idx,
                              int64_t nrows, double *o_rows, double *lse_rows, int nthreads)
{
    if (!q || !k || !v || !bh_idx || !row_idx || !o_rows || !lse_rows || nrows < 0 ||
        bad_rect(B, H, Nq, Nk, d, causal))
        return -1;
    for (int64_t t = 0; t < nrows; ++t)
        if (bh_idx[t] < 0 || bh_idx[t] >= B * H || row_idx[t] < 0 || row_idx[t] >= Nq) return -1;
    int failed = 0;
#pragma omp parallel num_threads(pick_threads(nthreads))
    {
        double *s_row = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s_row) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < nrows; ++t) {
            if (!s_row) continue;
            const int64_t bh = bh_idx[t], i = row_idx[t];
            const int64_t last = causal ? Nk - Nq + i : Nk - 1;
            attention_row_keys(q + (bh * Nq + i) * d, k + bh * Nk * d, v + bh * Nk * d, Nk, d, last,
                               scale, s_row, o_rows + t * d, lse_rows + t);
        }
        free(s_row);
    }
    return failed ? -2 : 0;
}

int oracle_max_threads(void)
{
    return pick_threads(0);
}

/* ------------------------------------------------------------------------
 * Backward pass: the gradients of the square attention above with respect
 * to q, k and v, given the gradient dO of a loss with respect to O.
 *
 * Sources: "Writing and Benchmarking Custom Kernels" (arunshar.com, ch. 10),
 * §10.3.2 "Backward-Pass Recomputation in FlashAttention": the softmax
 * backward of row i reduces to one scalar per query, D_i, the score
 * gradient is the probability times (dP minus that scalar), and
 * dL/dP_ij = dO_i . V_j.  The page's displayed formulas did not survive
 * extraction, so this is the textbook softmax/matrix-product chain rule,
 * which the surviving prose describes:
 *
 *     P_ij  = the two-pass softmax of the masked, scaled scores (as above)
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = dO_i . V_j
 *     D_i   = sum_j P_ij dP_ij          (equal to dO_i . O_i, the page's form)
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij K_j
 *     dK_j  = scale * sum_i dS_ij Q_i
 *
 * One head at a time: P and dS of the head are materialised (2 N^2
 * doubles), query rows are spread over threads for P, dS, D and dQ, then key
 * rows for dV and dK.  Inputs are bf16 bits (B, H, N, d) like the forward;
 * dq, dk, dv: B*H*N*d doubles; dsum (nullable): B*H*N doubles, the D_i.
 * Returns 0, -1 on bad arguments, -2 when the head's matrices cannot be
 * allocated.
 * ------------------------------------------------------------------------ */
int oracle_attn_bwd_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *dout, int64_t B, int64_t H, int64_t N, int64_t d,
                        int causal, double scale, double *dq, double *dk, double *dv,
                        double *dsum, int nthreads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || bad_shape(B, H, N, d)) return -1;
    const int64_t nd = N * d;
    double *P = (double *)malloc((size_t)(N * N) * sizeof(double));
    double *dS = (double *)malloc((size_t)(N * N) * sizeof(double));
    double *Qw = (double *)malloc((size_t)nd * sizeof(double));
    double *Kw = (double *)malloc((size_t)nd * sizeof(double));
    double *Vw = (double *)malloc((size_t)nd * sizeof(double));
    double *dOw = (double *)malloc((size_t)nd * sizeof(double));
    int failed = !P || !dS || !Qw || !Kw || !Vw || !dOw;
    for (int64_t bh = 0; bh < B * H && !failed; ++bh) {
        const int64_t base = bh * nd;
        for (int64_t t = 0; t < nd; ++t) {
            Qw[t] = bf16_bits_to_f64(q[base + t]);
            Kw[t] = bf16_bits_to_f64(k[base + t]);
            Vw[t] = bf16_bits_to_f64(v[base + t]);
            dOw[t] = bf16_bits_to_f64(dout[base + t]);
        }
#pragma omp parallel num_threads(pick_threads(nthreads))
        {
            double *dP = (double *)malloc((size_t)N * sizeof(double));
            if (!dP) {
#pragma omp atomic write
                failed = 1;
            }
            /* query rows: P, dP, D, dS and dQ */
#pragma omp for schedule(dynamic, 8)
            for (int64_t i = 0; i < N; ++i) {
                if (!dP) continue;
                double *Pi = P + i * N, *dSi = dS + i * N;
                const int64_t visible = causal ? i + 1 : N; /* keys 0 .. visible-1 */
                double m = -INFINITY;
                for (int64_t j = 0; j < visible; ++j) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += Qw[i * d + c] * Kw[j * d + c];
                    Pi[j] = scale * dot;
                    if (Pi[j] > m) m = Pi[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j < visible; ++j) {
                    Pi[j] = exp(Pi[j] - m);
                    l += Pi[j];
                }
                for (int64_t j = 0; j < visible; ++j) Pi[j] /= l;
                for (int64_t j = visible; j < N; ++j) Pi[j] = 0.0;
                double Di = 0.0;
                for (int64_t j = 0; j < visible; ++j) {
                    double g = 0.0;
                    for (int64_t c = 0; c < d; ++c) g += dOw[i * d + c] * Vw[j * d + c];
                    dP[j] = g;
                    Di += Pi[j] * g;
                }
                for (int64_t j = 0; j < N; ++j) dSi[j] = j < visible ? Pi[j] * (dP[j] - Di) : 0.0;
                if (dsum) dsum[bh * N + i] = Di;
                for (int64_t c = 0; c < d; ++c) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < visible; ++j) acc += dSi[j] * Kw[j * d + c];
                    dq[base + i * d + c] = scale * acc;
                }
            }
            /* key rows: dV and dK (column j of P and of dS) */
#pragma omp for schedule(dynamic, 8)
            for (int64_t j = 0; j < N; ++j) {
                for (int64_t c = 0; c < d; ++c) {
                    double gv = 0.0, gk = 0.0;
                    for (int64_t i = 0; i < N; ++i) {
                        gv += P[i * N + j] * dOw[i * d + c];
                        gk += dS[i * N + j] * Qw[i * d + c];
                    }
                    dv[base + j * d + c] = gv;
                    dk[base + j * d + c] = scale * gk;
                }
            }
            free(dP);
        }
    }
    free(P);
    free(dS);
    free(Qw);
    free(Kw);
    free(Vw);
    free(dOw);
    return failed ? -2 : 0;
}

/* ------------------------------------------------------------------------
 * Fused elementwise chain: bias add, GELU, dropout.
 *
 * Sources: "Fusion and IO-aware kernels" § The idea in one minute (a bias
 * add, a GELU and a dropout, each an HBM round trip when run separately) and
 * its fusion.py byte count; "Writing and Benchmarking Custom Kernels"
 * §10.2.1 (the tanh form of GELU the chapter's kernel computes).  For element
 * (r, c) of a rows x cols tensor, flat index e = r*cols + c:
 *
 *     h = x[r][c] + bias[c]
 *     g = 0.5 h (1 + tanh( sqrt(2/pi) (h + 0.044715 h^3) ))
 *     y = g / (1 - p)   if bit (e % 32) of keep[e / 32] is set, else 0
 *
 * The dropout draws are passed in as the packed keep mask (NULL: keep all).
 * x, bias: bf16 bits; y: rows*cols doubles.  Returns 0, -1 on bad arguments.
 * ------------------------------------------------------------------------ */
int oracle_bias_gelu_dropout_f64(const uint16_t *x, const uint16_t *bias, const uint32_t *keep,
                                 int64_t rows, int64_t cols, double p, double *y, int nthreads)
{
    if (!x || !bias || !y || rows < 1 || cols < 1 || !(p >= 0.0 && p < 1.0)) return -1;
    const double k0 = sqrt(2.0 / 3.14159265358979323846);
#pragma omp parallel for schedule(static) num_threads(pick_threads(nthreads))
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            const int64_t e = r * cols + c;
            const double h = bf16_bits_to_f64(x[e]) + bf16_bits_to_f64(bias[c]);
            const double g = 0.5 * h * (1.0 + tanh(k0 * (h + 0.044715 * h * h * h)));
            const int kept = keep ? (int)((keep[e >> 5] >> (e & 31)) & 1u) : 1;
            y[e] = kept ? g / (1.0 - p) : 0.0;
        }
    }
    return 0;
}
