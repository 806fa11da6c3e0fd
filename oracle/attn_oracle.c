/*
 * attn_oracle.c -- plain fp64 CPU attention: the oracle the CUDA path is checked against.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the benchmark's CPU-baseline
 * leg load this file's library.  The product path never calls it, and it shares no code,
 * header or constant with the CUDA library.
 *
 * What it computes is the plain definition of scaled-dot-product attention, written out
 * with explicit score rows, with no tiling, fusion or online rescaling:
 *
 *   S_ij  = sc * sum_k Q[i,k] K[j,k]          sc = scale, or 1/sqrt(d) when scale == 0
 *           ("AMD GPU에서도 동작하는 FlashAttention 구현체, Aule-Attention", API list:
 *            scale defaults to 1/sqrt(head_dim); Turing varlen article, flash_attn_torch.py
 *            docstring: softmax_scale None -> 1/sqrt(head_dim))
 *   S_ij  = -inf when causal and j > i         (Aule overview, "高性能实践" section: causal=True
 *                                                masks future tokens)
 *   P_ij  = exp(S_ij - m_i) / l_i,  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
 *           (FlashAttention-T review, 代码示例 示例2: max-subtracted softmax then P V)
 *   O_i   = sum_j P_ij V_j ;   LSE_i = m_i + ln l_i   (natural log of the scaled scores)
 *
 * GQA: query head h reads kv head g = h / (Hq/Hkv) (contiguous groups; Aule overview,
 * "支持多种注意力形式：GQA、MQA" section: 32 query heads over 8 kv heads, MQA = 1 kv head).
 *
 * Backward, analytic, for a given upstream gradient dO (FlashAttention-T review, 常见问题 4:
 * the backward recomputes the score matrix instead of storing it):
 *   dP_ij = dO_i . V_j ;  D_i = sum_j P_ij dP_ij ;  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = sc sum_j dS_ij K_j
 *   dK_j  = sc sum_{h in group(g)} sum_i dS_ij Q_i ;  dV_j = sum_{h in group(g)} sum_i P_ij dO_i
 *
 * It is computed in two plain passes: a row pass (per query row: S_i, P_i, O_i, LSE_i, D_i, dQ_i)
 * and a key pass (per key row j of a kv head: P_ij and dS_ij recomputed from LSE_i and D_i of
 * the row pass, then dK_j and dV_j).  Both passes are the definitions above evaluated term by term.
 *
 * Varlen (Turing varlen article, flash_attn_torch.py docstring): qkv is [T,3,H,d]; sequence s
 * is tokens [cu[s], cu[s+1]); each (sequence, head) is an independent attention problem with
 * indices relative to the sequence start; the output is [T,H,d] and LSE [H,T].
 *
 * Layouts: dense Q/O/dO/dQ [B,Hq,N,d], K/V/dK/dV [B,Hkv,N,d], LSE/D [B,Hq,N]; all contiguous.
 * Every function returns 0 on success and a negative value on a bad argument.
 *
 * Parity pins: see the tests for the oracle (closed forms, invariants, finite differences,
 * a library special case); no function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One attention problem: a single (query head, kv head) pair of n rows, addressed with
 * row strides so dense and varlen layouts share the same arithmetic. */
typedef struct {
    const double *q, *k, *v, *dout;  /* row r of X is X + r * stride */
    long q_stride, kv_stride, dout_stride;
    int n, d, causal;
    double sc;
} problem_t;

static double problem_score(const problem_t *p, int i, int j) {
    if (p->causal && j > i) return -INFINITY;
    const double *qi = p->q + (long)i * p->q_stride;
    const double *kj = p->k + (long)j * p->kv_stride;
    double acc = 0.0;
    for (int c = 0; c < p->d; ++c) acc += qi[c] * kj[c];
    return p->sc * acc;
}

/* Row pass for query row i.  s_row and p_row are scratch of length n.
 * Writes o_i (d values, may be NULL), *lse_i, and when dout is set, *D_i and dq_i. */
static void problem_row(const problem_t *p, int i, double *s_row, double *p_row,
                        double *o_i, double *lse_i, double *D_i, double *dq_i) {
    int n = p->n, d = p->d;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        s_row[j] = problem_score(p, i, j);
        if (s_row[j] > m) m = s_row[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j) l += exp(s_row[j] - m);
    for (int j = 0; j < n; ++j) p_row[j] = exp(s_row[j] - m) / l;
    if (lse_i) *lse_i = m + log(l);
    if (o_i) {
        for (int c = 0; c < d; ++c) o_i[c] = 0.0;
        for (int j = 0; j < n; ++j) {
            const double *vj = p->v + (long)j * p->kv_stride;
            for (int c = 0; c < d; ++c) o_i[c] += p_row[j] * vj[c];
        }
    }
    if (p->dout) {
        const double *doi = p->dout + (long)i * p->dout_stride;
        /* dP_ij = dO_i . V_j (stored in s_row, which is no longer needed) */
        for (int j = 0; j < n; ++j) {
            const double *vj = p->v + (long)j * p->kv_stride;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += doi[c] * vj[c];
            s_row[j] = acc;
        }
        double Dv = 0.0;
        for (int j = 0; j < n; ++j) Dv += p_row[j] * s_row[j];
        if (D_i) *D_i = Dv;
        if (dq_i) {
            for (int c = 0; c < d; ++c) dq_i[c] = 0.0;
            for (int j = 0; j < n; ++j) {
                double ds = p_row[j] * (s_row[j] - Dv);
                const double *kj = p->k + (long)j * p->kv_stride;
                for (int c = 0; c < d; ++c) dq_i[c] += p->sc * ds * kj[c];
            }
        }
    }
}

/* Key pass for key row j of one problem: adds this query head's terms to dk_j and dv_j,
 * using P_ij = exp(S_ij - LSE_i) and dS_ij = P_ij (dO_i . V_j - D_i). */
static void problem_key_accumulate(const problem_t *p, int j, const double *lse,
                                   long lse_stride, const double *Dvec, long D_stride,
                                   double *dk_j, double *dv_j) {
    int n = p->n, d = p->d;
    const double *vj = p->v + (long)j * p->kv_stride;
    for (int i = 0; i < n; ++i) {
        double s = problem_score(p, i, j);
        if (s == -INFINITY) continue; /* P_ij = 0: the term is exactly zero */
        double pij = exp(s - lse[(long)i * lse_stride]);
        const double *doi = p->dout + (long)i * p->dout_stride;
        const double *qi = p->q + (long)i * p->q_stride;
        double dp = 0.0;
        for (int c = 0; c < d; ++c) dp += doi[c] * vj[c];
        double ds = pij * (dp - Dvec[(long)i * D_stride]);
        for (int c = 0; c < d; ++c) {
            dv_j[c] += pij * doi[c];
            dk_j[c] += p->sc * ds * qi[c];
        }
    }
}

static double default_scale(double scale, int d) { return scale == 0.0 ? 1.0 / sqrt((double)d) : scale; }

static int check_dense(int B, int Hq, int Hkv, int N, int d, double scale) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if (!(scale >= 0.0)) return -1;
    return 0;
}

static problem_t dense_problem(const double *q, const double *k, const double *v,
                               const double *dout, int b, int h, int Hq, int Hkv, int N,
                               int d, int causal, double sc) {
    int G = Hq / Hkv, g = h / G;
    problem_t p;
    p.q = q + ((long)b * Hq + h) * N * d;
    p.k = k + ((long)b * Hkv + g) * N * d;
    p.v = v + ((long)b * Hkv + g) * N * d;
    p.dout = dout ? dout + ((long)b * Hq + h) * N * d : NULL;
    p.q_stride = d; p.kv_stride = d; p.dout_stride = d;
    p.n = N; p.d = d; p.causal = causal; p.sc = sc;
    return p;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Forward: O [B,Hq,N,d] and LSE [B,Hq,N] (either may be NULL). */
int oracle_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
               int B, int Hq, int Hkv, int N, int d, int causal, double scale) {
    if (check_dense(B, Hq, Hkv, N, d, scale)) return -1;
    double sc = default_scale(scale, d);
    long rows = (long)B * Hq * N;
    int err = 0;
#pragma omp parallel
    {
        double *s_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        double *p_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        if (!s_row || !p_row) err = 1;
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s_row || !p_row) continue;
            int i = (int)(r % N), bh = (int)(r / N), b = bh / Hq, h = bh % Hq;
            problem_t p = dense_problem(q, k, v, NULL, b, h, Hq, Hkv, N, d, causal, sc);
            problem_row(&p, i, s_row, p_row, o ? o + r * d : NULL, lse ? lse + r : NULL, NULL, NULL);
        }
        free(s_row); free(p_row);
    }
    return err ? -2 : 0;
}

/* Forward on selected rows only: rows[3*t..3*t+2] = (b, h, i).  o_rows [nrows,d], lse_rows [nrows]. */
int oracle_fwd_rows(const double *q, const double *k, const double *v, const int64_t *rows,
                    long nrows, double *o_rows, double *lse_rows, int B, int Hq, int Hkv,
                    int N, int d, int causal, double scale) {
    if (check_dense(B, Hq, Hkv, N, d, scale)) return -1;
    for (long t = 0; t < nrows; ++t)
        if (rows[3 * t] < 0 || rows[3 * t] >= B || rows[3 * t + 1] < 0 ||
            rows[3 * t + 1] >= Hq || rows[3 * t + 2] < 0 || rows[3 * t + 2] >= N) return -1;
    double sc = default_scale(scale, d);
    int err = 0;
#pragma omp parallel
    {
        double *s_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        double *p_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        if (!s_row || !p_row) err = 1;
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < nrows; ++t) {
            if (!s_row || !p_row) continue;
            problem_t p = dense_problem(q, k, v, NULL, (int)rows[3 * t], (int)rows[3 * t + 1],
                                        Hq, Hkv, N, d, causal, sc);
            problem_row(&p, (int)rows[3 * t + 2], s_row, p_row, o_rows + t * d, lse_rows + t,
                        NULL, NULL);
        }
        free(s_row); free(p_row);
    }
    return err ? -2 : 0;
}

/* Probabilities P [N,N] of one (b, h): for the invariant tests. */
int oracle_probs(const double *q, const double *k, double *P, int b, int h, int B, int Hq,
                 int Hkv, int N, int d, int causal, double scale) {
    if (check_dense(B, Hq, Hkv, N, d, scale) || b < 0 || b >= B || h < 0 || h >= Hq) return -1;
    double sc = default_scale(scale, d);
    problem_t p = dense_problem(q, k, k, NULL, b, h, Hq, Hkv, N, d, causal, sc);
    double *s_row = malloc(sizeof(double) * (N > 0 ? N : 1));
    if (!s_row) return -2;
    for (int i = 0; i < N; ++i) problem_row(&p, i, s_row, P + (long)i * N, NULL, NULL, NULL, NULL);
    free(s_row);
    return 0;
}

/* Row pass of the backward on all rows: LSE, D and dQ (each may be NULL). */
static int bwd_rows_all(const double *q, const double *k, const double *v, const double *dout,
                        double *lse, double *D, double *dq, int B, int Hq, int Hkv, int N, int d,
                        int causal, double sc) {
    long rows = (long)B * Hq * N;
    int err = 0;
#pragma omp parallel
    {
        double *s_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        double *p_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        if (!s_row || !p_row) err = 1;
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s_row || !p_row) continue;
            int i = (int)(r % N), bh = (int)(r / N), b = bh / Hq, h = bh % Hq;
            problem_t p = dense_problem(q, k, v, dout, b, h, Hq, Hkv, N, d, causal, sc);
            problem_row(&p, i, s_row, p_row, NULL, lse + r, D + r, dq ? dq + r * d : NULL);
        }
        free(s_row); free(p_row);
    }
    return err ? -2 : 0;
}

/* Full backward: dQ [B,Hq,N,d], dK and dV [B,Hkv,N,d] (dq may be NULL). */
int oracle_bwd(const double *q, const double *k, const double *v, const double *dout,
               double *dq, double *dk, double *dv, int B, int Hq, int Hkv, int N, int d,
               int causal, double scale) {
    if (check_dense(B, Hq, Hkv, N, d, scale) || !dout || !dk || !dv) return -1;
    double sc = default_scale(scale, d);
    long rows = (long)B * Hq * N;
    double *lse = malloc(sizeof(double) * (rows > 0 ? rows : 1));
    double *D = malloc(sizeof(double) * (rows > 0 ? rows : 1));
    if (!lse || !D) { free(lse); free(D); return -2; }
    int rc = bwd_rows_all(q, k, v, dout, lse, D, dq, B, Hq, Hkv, N, d, causal, sc);
    int G = Hq / Hkv;
    long keys = (long)B * Hkv * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < keys; ++r) {
        int j = (int)(r % N), bg = (int)(r / N), b = bg / Hkv, g = bg % Hkv;
        double *dk_j = dk + r * d, *dv_j = dv + r * d;
        for (int c = 0; c < d; ++c) { dk_j[c] = 0.0; dv_j[c] = 0.0; }
        for (int h = g * G; h < (g + 1) * G; ++h) {
            problem_t p = dense_problem(q, k, v, dout, b, h, Hq, Hkv, N, d, causal, sc);
            long base = ((long)b * Hq + h) * N;
            problem_key_accumulate(&p, j, lse + base, 1, D + base, 1, dk_j, dv_j);
        }
    }
    free(lse); free(D);
    return rc;
}

/* Backward on selected rows (dQ) and selected keys (dK, dV) of a large problem.
 * q_rows[3*t..] = (b, h, i) -> dq_rows [nq, d];  k_rows[3*t..] = (b, g, j) -> dk_rows, dv_rows [nk, d].
 * The row pass runs only over the query rows a selected key depends on (all rows of the
 * group's heads, or rows i >= j when causal). */
int oracle_bwd_sampled(const double *q, const double *k, const double *v, const double *dout,
                       const int64_t *q_rows, long nq, double *dq_rows,
                       const int64_t *k_rows, long nk, double *dk_rows, double *dv_rows,
                       int B, int Hq, int Hkv, int N, int d, int causal, double scale) {
    if (check_dense(B, Hq, Hkv, N, d, scale) || !dout) return -1;
    for (long t = 0; t < nq; ++t)
        if (q_rows[3 * t] < 0 || q_rows[3 * t] >= B || q_rows[3 * t + 1] < 0 ||
            q_rows[3 * t + 1] >= Hq || q_rows[3 * t + 2] < 0 || q_rows[3 * t + 2] >= N) return -1;
    for (long t = 0; t < nk; ++t)
        if (k_rows[3 * t] < 0 || k_rows[3 * t] >= B || k_rows[3 * t + 1] < 0 ||
            k_rows[3 * t + 1] >= Hkv || k_rows[3 * t + 2] < 0 || k_rows[3 * t + 2] >= N) return -1;
    double sc = default_scale(scale, d);
    int G = Hq / Hkv, err = 0;
    /* dQ rows: one row pass each. */
#pragma omp parallel
    {
        double *s_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        double *p_row = malloc(sizeof(double) * (N > 0 ? N : 1));
        if (!s_row || !p_row) err = 1;
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < nq; ++t) {
            if (!s_row || !p_row) continue;
            problem_t p = dense_problem(q, k, v, dout, (int)q_rows[3 * t], (int)q_rows[3 * t + 1],
                                        Hq, Hkv, N, d, causal, sc);
            double lse_i, D_i;
            problem_row(&p, (int)q_rows[3 * t + 2], s_row, p_row, NULL, &lse_i, &D_i,
                        dq_rows + t * d);
        }
        free(s_row); free(p_row);
    }
    if (err) return -2;
    /* dK/dV keys: LSE and D of every query row the key can see, then the key pass.
     * Rows below i0 never see key j under the causal mask (P_ij = 0 there); their LSE and D
     * slots stay NaN and are never read, because the key pass skips masked scores first. */
    for (long t = 0; t < nk; ++t) {
        int b = (int)k_rows[3 * t], g = (int)k_rows[3 * t + 1], j = (int)k_rows[3 * t + 2];
        int i0 = causal ? j : 0;
        long cnt = (long)G * N;
        double *lse = malloc(sizeof(double) * (cnt > 0 ? cnt : 1));
        double *D = malloc(sizeof(double) * (cnt > 0 ? cnt : 1));
        if (!lse || !D) { free(lse); free(D); return -2; }
        for (long r = 0; r < cnt; ++r) { lse[r] = NAN; D[r] = NAN; }
#pragma omp parallel
        {
            double *s_row = malloc(sizeof(double) * (N > 0 ? N : 1));
            double *p_row = malloc(sizeof(double) * (N > 0 ? N : 1));
            if (!s_row || !p_row) err = 1;
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < (long)G * (N - i0); ++r) {
                if (!s_row || !p_row) continue;
                int hh = (int)(r / (N - i0)), i = i0 + (int)(r % (N - i0));
                problem_t p = dense_problem(q, k, v, dout, b, g * G + hh, Hq, Hkv, N, d, causal, sc);
                problem_row(&p, i, s_row, p_row, NULL, lse + (long)hh * N + i,
                            D + (long)hh * N + i, NULL);
            }
            free(s_row); free(p_row);
        }
        double *dk_j = dk_rows + t * d, *dv_j = dv_rows + t * d;
        for (int c = 0; c < d; ++c) { dk_j[c] = 0.0; dv_j[c] = 0.0; }
        for (int hh = 0; hh < G && !err; ++hh) {
            problem_t p = dense_problem(q, k, v, dout, b, g * G + hh, Hq, Hkv, N, d, causal, sc);
            problem_key_accumulate(&p, j, lse + (long)hh * N, 1, D + (long)hh * N, 1, dk_j, dv_j);
        }
        free(lse); free(D);
        if (err) return -2;
    }
    return 0;
}

/* Varlen forward.  qkv [T,3,H,d], cu [nseq+1] (0-based prefix sums), out [T,H,d], lse [H,T]
 * (lse may be NULL).  Returns -1 when cu is not a valid prefix-sum array ending at T. */
int oracle_fwd_varlen(const double *qkv, const int32_t *cu, int nseq, int T, double *out,
                      double *lse, int H, int d, int causal, double scale) {
    if (nseq < 0 || T < 0 || H <= 0 || d <= 0 || !(scale >= 0.0) || !cu) return -1;
    if (cu[0] != 0 || cu[nseq] != T) return -1;
    for (int s = 0; s < nseq; ++s) if (cu[s + 1] < cu[s]) return -1;
    double sc = default_scale(scale, d);
    long tok = 3L * H * d; /* token stride of the packed tensor */
    long rows = (long)T * H;
    int err = 0;
#pragma omp parallel
    {
        int maxlen = 1;
        for (int s = 0; s < nseq; ++s) if (cu[s + 1] - cu[s] > maxlen) maxlen = cu[s + 1] - cu[s];
        double *s_row = malloc(sizeof(double) * maxlen);
        double *p_row = malloc(sizeof(double) * maxlen);
        if (!s_row || !p_row) err = 1;
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s_row || !p_row) continue;
            int t = (int)(r / H), h = (int)(r % H);
            int s = 0;
            while (!(cu[s] <= t && t < cu[s + 1])) ++s; /* sequence containing token t */
            int start = cu[s];
            problem_t p;
            p.q = qkv + (long)start * tok + 0L * H * d + (long)h * d;
            p.k = qkv + (long)start * tok + 1L * H * d + (long)h * d;
            p.v = qkv + (long)start * tok + 2L * H * d + (long)h * d;
            p.dout = NULL;
            p.q_stride = tok; p.kv_stride = tok; p.dout_stride = 0;
            p.n = cu[s + 1] - start; p.d = d; p.causal = causal; p.sc = sc;
            problem_row(&p, t - start, s_row, p_row, out + ((long)t * H + h) * d,
                        lse ? lse + (long)h * T + t : NULL, NULL, NULL);
        }
        free(s_row); free(p_row);
    }
    return err ? -2 : 0;
}

/* KV-cache (and cross-attention) forward: Nq queries against a cache of up to Nk keys per
 * (batch, kv head) (FlashAttention-T review, FAQ 4: at inference the KV cache is computed in
 * blocks; its practical advice 2: the prefill and decode phases).  q [B,Hq,Nq,d], k and v
 * [B,Hkv,Nk,d], lens [B] (NULL: every cache holds Nk keys; else 0 <= lens[b] <= Nk),
 * o [B,Hq,Nq,d], lse [B,Hq,Nq] (may be NULL).
 *
 * Query i of batch b sees the keys j < L = lens[b]; when causal, only j <= L - Nq + i: the
 * queries are the last Nq positions of a sequence of L tokens (bottom-right alignment; with
 * Nq == L it is the self-attention mask j <= i).  A row that sees no key has O = 0 and
 * LSE = -inf (the empty sum).  Otherwise the row is the plain softmax over its visible keys,
 * written out like the dense rows: explicit scores, max, sum, normalised weights. */
int oracle_fwd_kvcache(const double *q, const double *k, const double *v, const int32_t *lens,
                       double *o, double *lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                       int causal, double scale) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0 || Hq % Hkv != 0) return -1;
    if (!(scale >= 0.0)) return -1;
    if (lens)
        for (int b = 0; b < B; ++b) if (lens[b] < 0 || lens[b] > Nk) return -1;
    double sc = default_scale(scale, d);
    int G = Hq / Hkv;
    long rows = (long)B * Hq * Nq;
    int err = 0;
#pragma omp parallel
    {
        double *s_row = malloc(sizeof(double) * (Nk > 0 ? Nk : 1));
        if (!s_row) err = 1;
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s_row) continue;
            int i = (int)(r % Nq), bh = (int)(r / Nq), b = bh / Hq, h = bh % Hq, kvh = h / G;
            int L = lens ? lens[b] : Nk;
            int last = causal ? L - Nq + i : L - 1; /* last visible key */
            if (last > L - 1) last = L - 1;
            const double *qi = q + ((long)bh * Nq + i) * d;
            const double *kb = k + ((long)b * Hkv + kvh) * (long)Nk * d;
            const double *vb = v + ((long)b * Hkv + kvh) * (long)Nk * d;
            double *oi = o + r * d;
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            if (last < 0) {
                if (lse) lse[r] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int j = 0; j <= last; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += qi[c] * kb[(long)j * d + c];
                s_row[j] = sc * acc;
                if (s_row[j] > m) m = s_row[j];
            }
            double l = 0.0;
            for (int j = 0; j <= last; ++j) l += exp(s_row[j] - m);
            for (int j = 0; j <= last; ++j) {
                double pj = exp(s_row[j] - m) / l;
                for (int c = 0; c < d; ++c) oi[c] += pj * vb[(long)j * d + c];
            }
            if (lse) lse[r] = m + log(l);
        }
        free(s_row);
    }
    return err ? -2 : 0;
}

/* Backward of oracle_fwd_kvcache without cache lengths (cross-attention: Nq queries, Nk keys,
 * every cache full), with its bottom-right causal alignment: query i sees key j iff
 * j <= Nk - Nq + i when causal.  For an upstream gradient dout [B,Hq,Nq,d] it returns dq
 * [B,Hq,Nq,d] and dk, dv [B,Hkv,Nk,d] from the same analytic formulas as oracle_bwd
 * (dP_ij = dO_i . V_j, D_i = sum_j P_ij dP_ij, dS_ij = P_ij (dP_ij - D_i), dQ_i = sc sum_j
 * dS_ij K_j, dK_j = sc sum_i dS_ij Q_i, dV_j = sum_i P_ij dO_i over the query heads of the
 * group), written out per (batch, query head) with explicit P rows.  Rows that see no key
 * (Nq > Nk under the causal mask) have P = 0 and contribute nothing. */
int oracle_bwd_cross(const double *q, const double *k, const double *v, const double *dout, double *dq,
                     double *dk, double *dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     double scale) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0 || Hq % Hkv != 0) return -1;
    if (!(scale >= 0.0)) return -1;
    double sc = default_scale(scale, d);
    int G = Hq / Hkv;
    memset(dq, 0, sizeof(double) * (size_t)B * Hq * Nq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    int err = 0;
    /* one (batch, kv head) per task: its dk, dv rows are written by that task alone */
#pragma omp parallel
    {
        double *P = malloc(sizeof(double) * ((size_t)Nq * Nk + 1));
        double *dS = malloc(sizeof(double) * ((size_t)Nq * Nk + 1));
        if (!P || !dS) err = 1;
#pragma omp for schedule(dynamic, 1)
        for (long bg = 0; bg < (long)B * Hkv; ++bg) {
            if (!P || !dS) continue;
            int b = (int)(bg / Hkv), g = (int)(bg % Hkv);
            const double *kb = k + bg * (long)Nk * d, *vb = v + bg * (long)Nk * d;
            double *dkb = dk + bg * (long)Nk * d, *dvb = dv + bg * (long)Nk * d;
            for (int h = g * G; h < (g + 1) * G; ++h) {
                long qh = (long)b * Hq + h;
                const double *qb = q + qh * Nq * d, *dob = dout + qh * Nq * d;
                double *dqb = dq + qh * Nq * d;
                for (int i = 0; i < Nq; ++i) {
                    int last = causal ? Nk - Nq + i : Nk - 1;
                    if (last > Nk - 1) last = Nk - 1;
                    double *Pi = P + (long)i * Nk, *dSi = dS + (long)i * Nk;
                    double m = -INFINITY;
                    for (int j = 0; j < Nk; ++j) {
                        if (j > last) { Pi[j] = -INFINITY; continue; }
                        double acc = 0.0;
                        for (int c = 0; c < d; ++c) acc += qb[(long)i * d + c] * kb[(long)j * d + c];
                        Pi[j] = sc * acc;
                        if (Pi[j] > m) m = Pi[j];
                    }
                    double l = 0.0;
                    for (int j = 0; j <= last; ++j) l += exp(Pi[j] - m);
                    for (int j = 0; j < Nk; ++j) Pi[j] = (j <= last) ? exp(Pi[j] - m) / l : 0.0;
                    double Dv = 0.0;
                    for (int j = 0; j < Nk; ++j) {
                        double dp = 0.0;
                        for (int c = 0; c < d; ++c) dp += dob[(long)i * d + c] * vb[(long)j * d + c];
                        dSi[j] = dp;
                        Dv += Pi[j] * dp;
                    }
                    for (int j = 0; j < Nk; ++j) dSi[j] = Pi[j] * (dSi[j] - Dv);
                    for (int j = 0; j < Nk; ++j)
                        for (int c = 0; c < d; ++c) dqb[(long)i * d + c] += sc * dSi[j] * kb[(long)j * d + c];
                }
                for (int j = 0; j < Nk; ++j)
                    for (int i = 0; i < Nq; ++i) {
                        double pij = P[(long)i * Nk + j], dsij = dS[(long)i * Nk + j];
                        for (int c = 0; c < d; ++c) {
                            dvb[(long)j * d + c] += pij * dob[(long)i * d + c];
                            dkb[(long)j * d + c] += sc * dsij * qb[(long)i * d + c];
                        }
                    }
            }
        }
        free(P); free(dS);
    }
    return err ? -2 : 0;
}
