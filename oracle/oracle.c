/*
 * oracle.c -- plain, slow fp64 CPU reference for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the CPU-baseline leg of the bench
 * are the only callers. The CUDA path never links, loads or calls this file, and this file
 * shares no code, header or constant with it.
 *
 * Every input arrives as float64, widened exactly from the fp16/bf16 values the GPU reads.
 * All arithmetic is float64 with libm exp/log. There is no blocking, fusion or reordering
 * beyond what each function's source passage states.
 *
 * Sources (web pages, by title and section):
 *   [DEF]   "11. Fusion, recompute, and flash attention" (ml-compiler-from-scratch), section 11.2:
 *           S = Q K^T * scale, P = softmax(S) row by row, O = P V.
 *   [STAB]  ithelp.ithome.com.tw article 10405336, section "先回顧 Stable Softmax": subtract the
 *           row maximum m, p = exp(s - m), l = sum p, softmax = p / l.
 *   [ONL]   same chapter, section 11.6 "Online softmax": running (m_j, l_j, o_j), start from
 *           (-inf, 0, 0), correction factor exp(m_{j-1} - m_j), one division at the end.
 *   [BLK]   "Flash Attention 2" (linearalgebraforprogrammers.com), "Overview of the algorithm":
 *           the same recurrence one tile of b keys at a time, using the tile maximum.
 *   [MERGE] section 11.6, last paragraph, and exercise 3: merging two partial states.
 *   [LSE]   "Flash Attention 2", "Write the data back to HBM": L = m + log l per row.
 *   [CAUSAL] section 11.6 exercises ("query i may only attend to keys j <= i") and the
 *           "Attention" page of the phobos stdlib docs, "Causal attention".
 *   [BWD]   same chapter, section 11.9 ("Backward") and exercise "Backward with recompute":
 *           gradients from Q, K, V, dO with P recomputed.
 *   [ROPE]  the same "Attention" page, "Rotary position embeddings": `rope` (rotate-half) and
 *           `rope_pairs` (interleaved pairs).
 *
 * Masking reading: a key that does not exist (j >= Nk) or that causal masking hides (j > i) is
 * left out of every maximum and sum; it is never given a sentinel score.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_EMPTY_ROW = 2, ORACLE_ERR_NOMEM = 3 };

/* Number of keys query i may see: all Nk, or keys 0..i under causal masking [CAUSAL]. */
static int64_t visible_keys(int64_t i, int64_t nk, int causal) {
    if (!causal) return nk;
    return (i + 1 < nk) ? i + 1 : nk;
}

/* s = scale * (q . k) for one query row and one key row [DEF]. */
static double score(const double* q, const double* k, int64_t d, double scale) {
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += q[c] * k[c];
    return scale * acc;
}

/*
 * One query row, two passes [DEF][STAB]:
 *   scores s_j for the n visible keys; m = max s_j; p_j = exp(s_j - m); l = sum p_j;
 *   P_j = p_j / l; o = sum_j P_j v_j.  lse = m + log l [LSE].
 * `s` is caller-provided scratch of length >= n. P is written to `p_out` when non-null.
 */
static int two_pass_row(const double* q, const double* k, const double* v, int64_t n, int64_t d,
                        double scale, double* s, double* o, double* lse, double* p_out) {
    if (n <= 0) return ORACLE_ERR_EMPTY_ROW;
    for (int64_t j = 0; j < n; ++j) s[j] = score(q, k + j * d, d, scale);
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t j = 0; j < n; ++j) s[j] = s[j] / l;
    if (p_out)
        for (int64_t j = 0; j < n; ++j) p_out[j] = s[j];
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < n; ++j)
        for (int64_t c = 0; c < d; ++c) o[c] += s[j] * v[j * d + c];
    if (lse) *lse = m + log(l);
    return ORACLE_OK;
}

/*
 * Full attention over `bh` independent (batch, head) slices.
 *   q: [bh][nq][d], k, v: [bh][nk][d], out: [bh][nq][d], lse: [bh][nq] (may be NULL).
 * Rows are independent, so they are shared out over threads; each row is computed by
 * two_pass_row alone.
 */
int oracle_attention(const double* q, const double* k, const double* v, int64_t bh, int64_t nq,
                     int64_t nk, int64_t d, double scale, int causal, double* out, double* lse) {
    if (!q || !k || !v || !out || bh < 1 || nq < 1 || nk < 1 || d < 1) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)nk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < bh * nq; ++r) {
            if (!s) continue;
            int64_t h = r / nq, i = r % nq;
            int rc = two_pass_row(q + r * d, k + h * nk * d, v + h * nk * d,
                                  visible_keys(i, nk, causal), d, scale, s, out + r * d,
                                  lse ? lse + r : NULL, NULL);
            if (rc != ORACLE_OK) {
#pragma omp atomic write
                status = rc;
            }
        }
        free(s);
    }
    return status;
}

/*
 * Selected query rows of one (batch, head) slice, for sampled checks of large problems.
 *   q_rows: [n_rows][d], the rows of Q; row_pos[r]: that row's query position i (it decides
 *   causal visibility); k, v: [nk][d] of the same slice; out: [n_rows][d]; lse: [n_rows] or NULL.
 */
int oracle_attention_rows(const double* q_rows, const int64_t* row_pos, int64_t n_rows,
                          const double* k, const double* v, int64_t nk, int64_t d, double scale,
                          int causal, double* out, double* lse) {
    if (!q_rows || !row_pos || !k || !v || !out || n_rows < 0 || nk < 1 || d < 1)
        return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)nk * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            int rc = s ? two_pass_row(q_rows + r * d, k, v, visible_keys(row_pos[r], nk, causal),
                                      d, scale, s, out + r * d, lse ? lse + r : NULL, NULL)
                       : ORACLE_ERR_NOMEM;
            if (rc != ORACLE_OK) {
#pragma omp atomic write
                status = rc;
            }
        }
        free(s);
    }
    return status;
}

/*
 * The softmax matrix P = softmax(scale * Q K^T) of one slice, [nq][nk], with zeros where a
 * key is hidden [DEF][STAB]. For checking that every row of P is a probability distribution.
 */
int oracle_softmax(const double* q, const double* k, int64_t nq, int64_t nk, int64_t d,
                   double scale, int causal, double* p) {
    if (!q || !k || !p || nq < 1 || nk < 1 || d < 1) return ORACLE_ERR_ARG;
    double* s = (double*)malloc((size_t)nk * sizeof(double));
    double* o = (double*)malloc((size_t)d * sizeof(double));
    double* zero_v = (double*)calloc((size_t)(nk * d), sizeof(double));
    if (!s || !o || !zero_v) {
        free(s); free(o); free(zero_v);
        return ORACLE_ERR_NOMEM;
    }
    int status = ORACLE_OK;
    for (int64_t i = 0; i < nq && status == ORACLE_OK; ++i) {
        memset(p + i * nk, 0, (size_t)nk * sizeof(double));
        status = two_pass_row(q + i * d, k, zero_v, visible_keys(i, nk, causal), d, scale, s, o,
                              NULL, p + i * nk);
    }
    free(s); free(o); free(zero_v);
    return status;
}

/*
 * Online state of one query row over the keys [j0, j1) of one slice, taken `block` keys at a
 * time [ONL][BLK]. The state starts at m = -inf, l = 0, o = 0. For each block:
 *   m_new = max(m, max of the block's scores)
 *   corr  = exp(m - m_new)            (the state is empty while m = -inf: corr is 0 then)
 *   l     = l * corr + sum_j exp(s_j - m_new)
 *   o     = o * corr + sum_j exp(s_j - m_new) v_j
 *   m     = m_new
 * With block = 1 this is the per-key recurrence of section 11.6 exactly. The state is left
 * unnormalised: the answer is o / l.
 */
int oracle_online_state(const double* q, const double* k, const double* v, int64_t j0, int64_t j1,
                        int64_t d, double scale, int64_t block, double* m_out, double* l_out,
                        double* o) {
    if (!q || !k || !v || !m_out || !l_out || !o || j0 < 0 || j1 < j0 || d < 1 || block < 1)
        return ORACLE_ERR_ARG;
    double m = -INFINITY, l = 0.0;
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t start = j0; start < j1; start += block) {
        int64_t end = (start + block < j1) ? start + block : j1;
        double m_block = -INFINITY;
        for (int64_t j = start; j < end; ++j) {
            double s = score(q, k + j * d, d, scale);
            if (s > m_block) m_block = s;
        }
        double m_new = (m_block > m) ? m_block : m;
        double corr = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        l = l * corr;
        for (int64_t c = 0; c < d; ++c) o[c] = o[c] * corr;
        for (int64_t j = start; j < end; ++j) {
            double p = exp(score(q, k + j * d, d, scale) - m_new);
            l += p;
            for (int64_t c = 0; c < d; ++c) o[c] += p * v[j * d + c];
        }
        m = m_new;
    }
    *m_out = m;
    *l_out = l;
    return ORACLE_OK;
}

/*
 * Merge two partial states over disjoint key sets [MERGE]:
 *   m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m), o = o1 e^(m1-m) + o2 e^(m2-m).
 * An empty state (m = -inf, l = 0, o = 0) contributes nothing.
 */
int oracle_merge_state(double m1, double l1, const double* o1, double m2, double l2,
                       const double* o2, int64_t d, double* m_out, double* l_out, double* o) {
    if (!o1 || !o2 || !m_out || !l_out || !o || d < 1) return ORACLE_ERR_ARG;
    double m = (m1 > m2) ? m1 : m2;
    double f1 = (m1 == -INFINITY) ? 0.0 : exp(m1 - m);
    double f2 = (m2 == -INFINITY) ? 0.0 : exp(m2 - m);
    *m_out = m;
    *l_out = l1 * f1 + l2 * f2;
    for (int64_t c = 0; c < d; ++c) o[c] = o1[c] * f1 + o2[c] * f2;
    return ORACLE_OK;
}

/*
 * Full attention by the online recurrence, `block` keys at a time, then one division per row
 * [ONL][BLK]; lse = m + log l [LSE]. Independent of oracle_attention: the two share only the
 * dot product `score` and the visibility rule.
 */
int oracle_attention_online(const double* q, const double* k, const double* v, int64_t bh,
                            int64_t nq, int64_t nk, int64_t d, double scale, int causal,
                            int64_t block, double* out, double* lse) {
    if (!q || !k || !v || !out || bh < 1 || nq < 1 || nk < 1 || d < 1 || block < 1)
        return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t r = 0; r < bh * nq; ++r) {
        int64_t h = r / nq, i = r % nq;
        int64_t n = visible_keys(i, nk, causal);
        double m, l;
        double* o = out + r * d;
        int rc = (n > 0) ? oracle_online_state(q + r * d, k + h * nk * d, v + h * nk * d, 0, n, d,
                                               scale, block, &m, &l, o)
                         : ORACLE_ERR_EMPTY_ROW;
        if (rc != ORACLE_OK) {
#pragma omp atomic write
            status = rc;
            continue;
        }
        for (int64_t c = 0; c < d; ++c) o[c] = o[c] / l;
        if (lse) lse[r] = m + log(l);
    }
    return status;
}

/*
 * Gradients of the attention forward [BWD]. With P = softmax(scale * Q K^T) row by row (hidden
 * keys have P = 0) and O = P V, and an upstream gradient dO of the loss with respect to O:
 *   dV = P^T dO
 *   dP = dO V^T
 *   dS = P * (dP - rowsum(dO * O))        (elementwise; rowsum over the head dimension)
 *   dQ = scale * dS K,   dK = scale * dS^T Q
 * The pages name the backward pass and its recompute of P from Q, K and the log-sum-exp, but
 * print no formulas; these are the derivative of the forward definition [DEF], taken plainly.
 *   q, dout: [bh][nq][d]; k, v: [bh][nk][d]; dq: [bh][nq][d]; dk, dv: [bh][nk][d].
 */
int oracle_attention_backward(const double* q, const double* k, const double* v,
                              const double* dout, int64_t bh, int64_t nq, int64_t nk, int64_t d,
                              double scale, int causal, double* dq, double* dk, double* dv) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || bh < 1 || nq < 1 || nk < 1 || d < 1)
        return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t h = 0; h < bh; ++h) {
        const double* qh = q + h * nq * d;
        const double* kh = k + h * nk * d;
        const double* vh = v + h * nk * d;
        const double* doh = dout + h * nq * d;
        double* dqh = dq + h * nq * d;
        double* dkh = dk + h * nk * d;
        double* dvh = dv + h * nk * d;
        double* p = (double*)calloc((size_t)(nq * nk), sizeof(double));
        double* s = (double*)malloc((size_t)nk * sizeof(double));
        double* o = (double*)malloc((size_t)d * sizeof(double));
        if (!p || !s || !o) {
            free(p); free(s); free(o);
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
            continue;
        }
        for (int64_t i = 0; i < nq * d; ++i) dqh[i] = 0.0;
        for (int64_t i = 0; i < nk * d; ++i) dkh[i] = dvh[i] = 0.0;
        for (int64_t i = 0; i < nq; ++i) {
            const int64_t n = visible_keys(i, nk, causal);
            int rc = two_pass_row(qh + i * d, kh, vh, n, d, scale, s, o, NULL, p + i * nk);
            if (rc != ORACLE_OK) {
#pragma omp atomic write
                status = rc;
                break;
            }
            double delta = 0.0;  /* rowsum(dO * O) */
            for (int64_t c = 0; c < d; ++c) delta += doh[i * d + c] * o[c];
            for (int64_t j = 0; j < n; ++j) {
                const double pij = p[i * nk + j];
                double dp = 0.0;
                for (int64_t c = 0; c < d; ++c) dp += doh[i * d + c] * vh[j * d + c];
                const double ds = pij * (dp - delta);
                for (int64_t c = 0; c < d; ++c) {
                    dvh[j * d + c] += pij * doh[i * d + c];
                    dqh[i * d + c] += scale * ds * kh[j * d + c];
                    dkh[j * d + c] += scale * ds * qh[i * d + c];
                }
            }
        }
        free(p); free(s); free(o);
    }
    return status;
}

/*
 * Rotary position embedding of rows of width d, in place [ROPE]:
 *   form 0, rotate-half (phobos "Attention", `rope`): row = [a | b] with halves a, b of d/2;
 *     a' = a cos - b sin,  b' = b cos + a sin   (element i of a pairs with element i of b)
 *   form 1, interleaved pairs (`rope_pairs`): elements 2i and 2i+1 form the pair (x0, x1);
 *     x0' = x0 cos - x1 sin,  x1' = x1 cos + x0 sin
 * x: [rows][d]; cos_t, sin_t: [rows][d/2], the angle of pair i of each row. Both halves are read
 * before either is written.
 */
int oracle_rope(double* x, const double* cos_t, const double* sin_t, int64_t rows, int64_t d,
                int form) {
    if (!x || !cos_t || !sin_t || rows < 0 || d < 2 || d % 2 != 0 || (form != 0 && form != 1))
        return ORACLE_ERR_ARG;
    const int64_t h = d / 2;
    for (int64_t r = 0; r < rows; ++r) {
        double* row = x + r * d;
        for (int64_t i = 0; i < h; ++i) {
            const int64_t i0 = (form == 0) ? i : 2 * i;
            const int64_t i1 = (form == 0) ? i + h : 2 * i + 1;
            const double x0 = row[i0], x1 = row[i1];
            const double c = cos_t[r * h + i], sn = sin_t[r * h + i];
            row[i0] = x0 * c - x1 * sn;
            row[i1] = x1 * c + x0 * sn;
        }
    }
    return ORACLE_OK;
}

/* Threads an OpenMP region of this library would use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
