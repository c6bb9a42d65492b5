/*
 * fa_oracle.c -- plain, slow, FP64 CPU oracle for exact attention (forward
 * and its gradients).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [FA3H]  "FlashAttention-3 on Hopper" (l1-ca0.github.io):
 *           sec. 3.1 scaled dot-product attention with masks as -inf,
 *           sec. 3.2 safe softmax and the streaming state (m, l, O~),
 *           sec. 3.2.1 block-combine, sec. 4.2 online-softmax invariant,
 *           sec. 4.6 finalize: empty rows give O = 0 and LSE = -inf,
 *           sec. 4.7 causal predicate col > row + (Nk - Nq),
 *           sec. 7.1 gradient math (product rule through S = alpha Q K^T
 *           and O = P V; softmax Jacobian contracted to D_i = <P_i, dP_i>),
 *           sec. 6.3 block quantization, sec. 6.4 incoherent processing
 *           M = (1/sqrt d) H D with H a Hadamard matrix, D = diag(+-1).
 *   [FAv4]  "FlashAttention v1-v4: from IO awareness to asynchronous
 *           pipelines" (tom-jerr.github.io), section on the common
 *           computation graph (m_j, alpha_j, P~_j, l_j, U_j recurrence) and
 *           section "conditional rescale" (reference point r, threshold tau,
 *           LSE = r ln2 + ln l_r).
 *   [FA3A]  "03 FA3: Hopper asynchrony and overlap" (llm-infra-atlas), sec. 4
 *           FP8: per-tile scales folded into the softmax scale; sec. 5
 *           softcap s' = c tanh(s / c) on the scaled scores.
 *   Variants ([FA3H] sec. 4.6 learnable sinks folded into the row sum,
 *           sec. 4.7 local (sliding-window) masks with a left boundary,
 *           and the order transform-then-mask).
 *
 * Layout conventions (chosen by this library, stated in include/fa.h):
 *   Q, K, V, O rows are addressed through a leading dimension (element
 *   stride between consecutive sequence positions), so that one head of a
 *   [B][N][H][d] tensor is passed as base + (b*N*H + h)*d with ld = H*d.
 *
 * Build: plain C11, -O2 -ffp-contract=off (no FMA contraction, so x86-64
 * and aarch64 hosts produce identical bits), -lm -lpthread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Plain definition, one head: [FA3H] sec. 3.1 (attention), sec. 3.2 (safe   */
/* softmax: subtract the row maximum), sec. 4.6 (LSE in natural-log units,   */
/* empty rows), sec. 4.7 (causal predicate, bottom-right aligned).           */
/*                                                                           */
/* For every requested query row i:                                          */
/*   S_ij = alpha * sum_k q_ik k_jk            (j visible; else -inf)        */
/*   m_i  = max_j S_ij                                                       */
/*   P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)                          */
/*   O_i  = sum_j P_ij v_j                                                   */
/*   LSE_i = m_i + log(sum_j exp(S_ij - m_i))                                */
/* A row with no visible key gets O_i = 0 and LSE_i = -inf.                   */
/* The row of S and of P is materialised in full (length Nk).                */
/* ------------------------------------------------------------------------ */

static int visible(int i, int j, int Nq, int Nk, int causal)
{
    if (!causal) return 1;
    /* masked when col > row + (Nk - Nq) */
    return !((long)j > (long)i + ((long)Nk - (long)Nq));
}

/* Computes one query row.  s and p are caller scratch of length Nk. */
static void attention_row(const double *q, const double *k, const double *v,
                          int i, int Nq, int Nk, int d, long ldk, long ldv,
                          double alpha, int causal, double *s, double *p,
                          double *o_row, double *lse_out, double *probs_row)
{
    double m = -INFINITY;
    for (int j = 0; j < Nk; ++j) {
        if (visible(i, j, Nq, Nk, causal)) {
            double dot = 0.0;
            const double *kj = k + (long)j * ldk;
            for (int c = 0; c < d; ++c) dot += q[c] * kj[c];
            s[j] = alpha * dot;
        } else {
            s[j] = -INFINITY;
        }
        if (s[j] > m) m = s[j];
    }
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    if (m == -INFINITY) {               /* empty row: [FA3H] sec. 4.6 */
        *lse_out = -INFINITY;
        if (probs_row)
            for (int j = 0; j < Nk; ++j) probs_row[j] = 0.0;
        return;
    }
    double l = 0.0;
    for (int j = 0; j < Nk; ++j) {
        p[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
        l += p[j];
    }
    for (int j = 0; j < Nk; ++j) p[j] /= l;        /* normalised P row */
    for (int j = 0; j < Nk; ++j) {
        if (p[j] == 0.0) continue;
        const double *vj = v + (long)j * ldv;
        for (int c = 0; c < d; ++c) o_row[c] += p[j] * vj[c];
    }
    *lse_out = m + log(l);
    if (probs_row)
        for (int j = 0; j < Nk; ++j) probs_row[j] = p[j];
}

/*
 * oracle_attention_head: one (batch, head).  rows == NULL means every row
 * 0..Nq-1 (o row r at o + r*ldo, lse[r]); otherwise only rows[0..n_rows)
 * are computed and written at o + t*ldo, lse[t] for t = 0..n_rows-1.
 * probs (optional, Nq x Nk row-major, only with rows == NULL) receives P.
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
int oracle_attention_head(const double *q, const double *k, const double *v,
                          int Nq, int Nk, int d, long ldq, long ldk, long ldv,
                          double alpha, int causal, const int *rows, int n_rows,
                          double *o, long ldo, double *lse, double *probs)
{
    if (Nq < 0 || Nk < 0 || d < 1 || !q || !k || !v || !o || !lse) return -1;
    if (rows && probs) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    if (!s || !p) { free(s); free(p); return -1; }
    int count = rows ? n_rows : Nq;
    for (int t = 0; t < count; ++t) {
        int i = rows ? rows[t] : t;
        if (i < 0 || i >= Nq) { free(s); free(p); return -1; }
        attention_row(q + (long)i * ldq, k, v, i, Nq, Nk, d, ldk, ldv, alpha,
                      causal, s, p, o + (long)t * ldo, &lse[t],
                      probs ? probs + (long)t * Nk : NULL);
    }
    free(s);
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Whole tensors, [B][N][H][d] for Q/K/V/O and [B][H][N] for LSE, threaded   */
/* over (b, h, block of FWD_ROWS query rows).  Rows are independent          */
/* ([FA3H] sec. 3.4.2), and each row is computed by attention_row alone, so  */
/* the split changes no bit of the result; it only keeps every core busy     */
/* when B * H is small (one long sequence of few heads).                     */
/* ------------------------------------------------------------------------ */

#define FWD_ROWS 256

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int B, H, N, d, causal;
    double alpha;
    int next;              /* work counter, guarded by mu */
    int err;
    pthread_mutex_t mu;
} fwd_job;

static void *fwd_worker(void *arg)
{
    fwd_job *J = (fwd_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int u = J->next++;
        pthread_mutex_unlock(&J->mu);
        const int nblk = (J->N + FWD_ROWS - 1) / FWD_ROWS;
        if (u >= J->B * J->H * nblk) break;
        int blk = u % nblk, bh = u / nblk;
        int b = bh / J->H, h = bh % J->H;
        long ld = (long)J->H * J->d;
        long off = ((long)b * J->N * J->H + h) * J->d;
        int r0 = blk * FWD_ROWS;
        int nr = J->N - r0 < FWD_ROWS ? J->N - r0 : FWD_ROWS;
        int rows[FWD_ROWS];
        for (int t = 0; t < nr; ++t) rows[t] = r0 + t;
        /* rows r0 .. r0+nr-1 are written at o + (r0 + t) ld, lse[r0 + t] */
        int rc = oracle_attention_head(J->q + off, J->k + off, J->v + off,
                                       J->N, J->N, J->d, ld, ld, ld, J->alpha,
                                       J->causal, rows, nr, J->o + off + (long)r0 * ld, ld,
                                       J->lse + ((long)b * J->H + h) * J->N + r0,
                                       NULL);
        if (rc) {
            pthread_mutex_lock(&J->mu);
            J->err = rc;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

int oracle_attention_fwd(const double *q, const double *k, const double *v,
                         double *o, double *lse, int B, int H, int N, int d,
                         double alpha, int causal, int n_threads)
{
    if (B < 1 || H < 1 || N < 0 || d < 1) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    fwd_job J = {q, k, v, o, lse, B, H, N, d, causal, alpha, 0, 0,
                 PTHREAD_MUTEX_INITIALIZER};
    pthread_t th[512];
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&th[t], NULL, fwd_worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) fwd_worker(&J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    return J.err;
}

/* ------------------------------------------------------------------------ */
/* Score and mask variants, one head ([FA3H] sec. 4.6 "learnable sinks",     */
/* sec. 4.7 local attention and the rule that a score transformation comes   */
/* before the final mask; [FA3A] sec. 5 softcap).                            */
/*                                                                           */
/* Visibility, with the diagonal bottom-right aligned, diag = i + (Nk - Nq): */
/*   key j is hidden from query i when j > diag + wr (right window, wr >= 0) */
/*   or when j < diag - wl (left window, wl >= 0); -1 means no bound on that */
/*   side.  (wl, wr) = (-1, 0) is the causal mask, (-1, -1) no mask.         */
/* Scores, for visible keys only (so the transform never sees a masked       */
/* entry, which is the transform-then-mask order):                          */
/*   S_ij = alpha q_i . k_j;  softcap c > 0:  S_ij <- c tanh(S_ij / c).      */
/* Sink: one extra logit sigma per row that joins the softmax denominator    */
/* and carries no value:                                                     */
/*   m_i  = max(max_j S_ij, sigma)                                           */
/*   l_i  = sum_j exp(S_ij - m_i) + exp(sigma - m_i)                         */
/*   O_i  = sum_j exp(S_ij - m_i) v_j / l_i,  LSE_i = m_i + log l_i.         */
/* Without a sink, a row with no visible key gets O = 0 and LSE = -inf; with */
/* one it gets O = 0 and LSE = sigma.                                        */
/* ------------------------------------------------------------------------ */

static int visible_ext(int i, int j, int Nq, int Nk, int wl, int wr)
{
    long diag = (long)i + ((long)Nk - (long)Nq);
    if (wr >= 0 && (long)j > diag + wr) return 0;
    if (wl >= 0 && (long)j < diag - wl) return 0;
    return 1;
}

static void attention_row_ext(const double *q, const double *k, const double *v,
                              int i, int Nq, int Nk, int d, long ldk, long ldv,
                              double alpha, int wl, int wr, double softcap,
                              int has_sink, double sink, double *s,
                              double *o_row, double *lse_out)
{
    double m = has_sink ? sink : -INFINITY;
    for (int j = 0; j < Nk; ++j) {
        if (visible_ext(i, j, Nq, Nk, wl, wr)) {
            double dot = 0.0;
            const double *kj = k + (long)j * ldk;
            for (int c = 0; c < d; ++c) dot += q[c] * kj[c];
            double x = alpha * dot;
            if (softcap > 0.0) x = softcap * tanh(x / softcap);
            s[j] = x;
        } else {
            s[j] = -INFINITY;
        }
        if (s[j] > m) m = s[j];
    }
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    if (m == -INFINITY) {               /* no visible key and no sink */
        *lse_out = -INFINITY;
        return;
    }
    double l = has_sink ? exp(sink - m) : 0.0;
    for (int j = 0; j < Nk; ++j) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - m);
        l += p;
        const double *vj = v + (long)j * ldv;
        for (int c = 0; c < d; ++c) o_row[c] += p * vj[c];
    }
    for (int c = 0; c < d; ++c) o_row[c] /= l;
    *lse_out = m + log(l);
}

/*
 * oracle_attention_ext_head: one (batch, head) with the variants above.
 * sink == NULL: no sink; otherwise *sink is this head's sigma.  rows as in
 * oracle_attention_head.  Returns 0, or -1 on a bad argument (softcap < 0,
 * a window bound below -1) or an allocation failure.
 */
int oracle_attention_ext_head(const double *q, const double *k, const double *v,
                              int Nq, int Nk, int d, long ldq, long ldk, long ldv,
                              double alpha, int wl, int wr, double softcap,
                              const double *sink, const int *rows, int n_rows,
                              double *o, long ldo, double *lse)
{
    if (Nq < 0 || Nk < 0 || d < 1 || !q || !k || !v || !o || !lse) return -1;
    if (wl < -1 || wr < -1 || !(softcap >= 0.0)) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    if (!s) return -1;
    int count = rows ? n_rows : Nq;
    for (int t = 0; t < count; ++t) {
        int i = rows ? rows[t] : t;
        if (i < 0 || i >= Nq) { free(s); return -1; }
        attention_row_ext(q + (long)i * ldq, k, v, i, Nq, Nk, d, ldk, ldv, alpha,
                          wl, wr, softcap, sink != NULL, sink ? *sink : 0.0, s,
                          o + (long)t * ldo, &lse[t]);
    }
    free(s);
    return 0;
}

typedef struct {
    const double *q, *k, *v, *sinks;
    double *o, *lse;
    int B, H, N, d, wl, wr;
    double alpha, softcap;
    int next;
    int err;
    pthread_mutex_t mu;
} ext_job;

static void *ext_worker(void *arg)
{
    ext_job *J = (ext_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int u = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (u >= J->B * J->H) break;
        int b = u / J->H, h = u % J->H;
        long ld = (long)J->H * J->d;
        long off = ((long)b * J->N * J->H + h) * J->d;
        int rc = oracle_attention_ext_head(J->q + off, J->k + off, J->v + off,
                                           J->N, J->N, J->d, ld, ld, ld, J->alpha,
                                           J->wl, J->wr, J->softcap,
                                           J->sinks ? J->sinks + h : NULL, NULL, 0,
                                           J->o + off, ld,
                                           J->lse + ((long)b * J->H + h) * J->N);
        if (rc) {
            pthread_mutex_lock(&J->mu);
            J->err = rc;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

/* Whole [B][N][H][d] tensors with the variants; sinks: NULL or sigma per
 * head, [H]. */
int oracle_attention_ext_fwd(const double *q, const double *k, const double *v,
                             double *o, double *lse, int B, int H, int N, int d,
                             double alpha, int wl, int wr, double softcap,
                             const double *sinks, int n_threads)
{
    if (B < 1 || H < 1 || N < 0 || d < 1) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    ext_job J = {q, k, v, sinks, o, lse, B, H, N, d, wl, wr, alpha, softcap, 0, 0,
                 PTHREAD_MUTEX_INITIALIZER};
    pthread_t th[512];
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&th[t], NULL, ext_worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) ext_worker(&J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    return J.err;
}

/* ------------------------------------------------------------------------ */
/* Gradients, one head: [FA3H] sec. 7.1.  With S = alpha Q K^T (masked       */
/* entries -inf), P = softmax(S) row-wise and O = P V, for an upstream       */
/* gradient dO:                                                              */
/*   dV  = P^T dO                                                            */
/*   dP  = dO V^T                                                            */
/*   D_i = sum_j P_ij dP_ij          (the softmax Jacobian, contracted)      */
/*   dS  = P o (dP - D)              (o: elementwise; D broadcast per row)   */
/*   dQ  = alpha dS K,   dK = alpha dS^T Q                                   */
/* P is materialised row by row from the definition above; a row with no     */
/* visible key contributes nothing.  dq rows: every query row; dk, dv rows:  */
/* every key row (accumulated over the query rows).                          */
/* ------------------------------------------------------------------------ */
int oracle_attention_bwd_head(const double *q, const double *k, const double *v,
                              const double *dout, int Nq, int Nk, int d,
                              long ldq, long ldk, long ldv, long lddo,
                              double alpha, int causal, double *dq, long lddq,
                              double *dk, long lddk, double *dv, long lddv)
{
    if (Nq < 0 || Nk < 0 || d < 1 || !q || !k || !v || !dout || !dq || !dk || !dv)
        return -1;
    size_t nk1 = (size_t)(Nk > 0 ? Nk : 1);
    double *s = (double *)malloc(sizeof(double) * nk1);
    double *p = (double *)malloc(sizeof(double) * nk1);
    double *pr = (double *)malloc(sizeof(double) * nk1);
    double *dp = (double *)malloc(sizeof(double) * nk1);
    double *orow = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !p || !pr || !dp || !orow) {
        free(s); free(p); free(pr); free(dp); free(orow);
        return -1;
    }
    for (int j = 0; j < Nk; ++j)
        for (int c = 0; c < d; ++c) {
            dk[(long)j * lddk + c] = 0.0;
            dv[(long)j * lddv + c] = 0.0;
        }
    for (int i = 0; i < Nq; ++i) {
        const double *qi = q + (long)i * ldq;
        const double *doi = dout + (long)i * lddo;
        double *dqi = dq + (long)i * lddq;
        double lse;
        attention_row(qi, k, v, i, Nq, Nk, d, ldk, ldv, alpha, causal, s, p,
                      orow, &lse, pr);
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        if (lse == -INFINITY) continue;          /* no visible key */
        /* dP_ij = dO_i . v_j ; D_i = sum_j P_ij dP_ij */
        double D = 0.0;
        for (int j = 0; j < Nk; ++j) {
            const double *vj = v + (long)j * ldv;
            double t = 0.0;
            for (int c = 0; c < d; ++c) t += doi[c] * vj[c];
            dp[j] = t;
            D += pr[j] * t;
        }
        for (int j = 0; j < Nk; ++j) {
            if (pr[j] == 0.0) continue;
            const double ds = pr[j] * (dp[j] - D);
            const double *kj = k + (long)j * ldk;
            double *dkj = dk + (long)j * lddk;
            double *dvj = dv + (long)j * lddv;
            for (int c = 0; c < d; ++c) {
                dqi[c] += alpha * ds * kj[c];
                dkj[c] += alpha * ds * qi[c];
                dvj[c] += pr[j] * doi[c];
            }
        }
    }
    free(s); free(p); free(pr); free(dp); free(orow);
    return 0;
}

typedef struct {
    const double *q, *k, *v, *dout;
    double *dq, *dk, *dv;
    int B, H, N, d, causal;
    double alpha;
    int next;
    int err;
    pthread_mutex_t mu;
} bwd_job;

static void *bwd_worker(void *arg)
{
    bwd_job *J = (bwd_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int u = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (u >= J->B * J->H) break;
        int b = u / J->H, h = u % J->H;
        long ld = (long)J->H * J->d;
        long off = ((long)b * J->N * J->H + h) * J->d;
        int rc = oracle_attention_bwd_head(J->q + off, J->k + off, J->v + off,
                                           J->dout + off, J->N, J->N, J->d, ld,
                                           ld, ld, ld, J->alpha, J->causal,
                                           J->dq + off, ld, J->dk + off, ld,
                                           J->dv + off, ld);
        if (rc) {
            pthread_mutex_lock(&J->mu);
            J->err = rc;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

/* Whole [B][N][H][d] tensors, threaded over (b, h): each head's gradients
 * depend on that head alone. */
int oracle_attention_bwd(const double *q, const double *k, const double *v,
                         const double *dout, double *dq, double *dk, double *dv,
                         int B, int H, int N, int d, double alpha, int causal,
                         int n_threads)
{
    if (B < 1 || H < 1 || N < 0 || d < 1) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    bwd_job J = {q, k, v, dout, dq, dk, dv, B, H, N, d, causal, alpha, 0, 0,
                 PTHREAD_MUTEX_INITIALIZER};
    pthread_t th[512];
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&th[t], NULL, bwd_worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) bwd_worker(&J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    return J.err;
}


/* ------------------------------------------------------------------------ */
/* Gradients of the variants, one head: [FA3H] sec. 7.1 applied to the      */
/* definition of the variants above.  With u_ij = alpha q_i.k_j, the score   */
/* S_ij = u_ij (no softcap) or c tanh(u_ij / c), P_ij = exp(S_ij - LSE_i)    */
/* over visible keys and the sink's share P_i,sink = exp(sigma - LSE_i):     */
/*   dV_j  = sum_i P_ij dO_i,   dP_ij = dO_i . v_j,                          */
/*   D_i   = sum_j P_ij dP_ij   (the sink has no value: dP_i,sink = 0)       */
/*   dS_ij = P_ij (dP_ij - D_i),  dU_ij = dS_ij dS/du = dS_ij (1 - t_ij^2)   */
/*           with t_ij = tanh(u_ij / c) (softcap), else dU = dS              */
/*   dQ_i  = alpha sum_j dU_ij k_j,  dK_j = alpha sum_i dU_ij q_i            */
/*   dsigma = sum_i P_i,sink (0 - D_i) = -sum_i P_i,sink D_i                  */
/* dsink (optional) receives dsigma of this head.  Rows with neither a       */
/* visible key nor a sink contribute nothing.                                */
/* ------------------------------------------------------------------------ */
int oracle_attention_bwd_ext_head(const double *q, const double *k, const double *v,
                                  const double *dout, int Nq, int Nk, int d,
                                  double alpha, int wl, int wr, double softcap,
                                  const double *sink, double *dq, double *dk,
                                  double *dv, double *dsink)
{
    if (Nq < 0 || Nk < 0 || d < 1 || !q || !k || !v || !dout || !dq || !dk || !dv)
        return -1;
    if (wl < -1 || wr < -1 || !(softcap >= 0.0)) return -1;
    size_t nk1 = (size_t)(Nk > 0 ? Nk : 1);
    double *s = (double *)malloc(sizeof(double) * nk1);
    double *t = (double *)malloc(sizeof(double) * nk1);
    double *p = (double *)malloc(sizeof(double) * nk1);
    double *dp = (double *)malloc(sizeof(double) * nk1);
    if (!s || !t || !p || !dp) { free(s); free(t); free(p); free(dp); return -1; }
    for (long x = 0; x < (long)Nk * d; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
    double ds_sink = 0.0;
    for (int i = 0; i < Nq; ++i) {
        const double *qi = q + (long)i * d, *doi = dout + (long)i * d;
        double *dqi = dq + (long)i * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        double m = sink ? *sink : -INFINITY;
        for (int j = 0; j < Nk; ++j) {
            s[j] = -INFINITY;
            t[j] = 0.0;
            if (!visible_ext(i, j, Nq, Nk, wl, wr)) continue;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qi[c] * k[(long)j * d + c];
            double u = alpha * dot;
            if (softcap > 0.0) { t[j] = tanh(u / softcap); s[j] = softcap * t[j]; }
            else s[j] = u;
            if (s[j] > m) m = s[j];
        }
        if (m == -INFINITY) continue;
        double l = sink ? exp(*sink - m) : 0.0;
        for (int j = 0; j < Nk; ++j) {
            p[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
            l += p[j];
        }
        for (int j = 0; j < Nk; ++j) p[j] /= l;
        double D = 0.0;
        for (int j = 0; j < Nk; ++j) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += doi[c] * v[(long)j * d + c];
            dp[j] = acc;
            D += p[j] * acc;
        }
        if (sink) ds_sink -= exp(*sink - m) / l * D;
        for (int j = 0; j < Nk; ++j) {
            if (p[j] == 0.0) continue;
            double du = p[j] * (dp[j] - D);
            if (softcap > 0.0) du *= 1.0 - t[j] * t[j];
            for (int c = 0; c < d; ++c) {
                dqi[c] += alpha * du * k[(long)j * d + c];
                dk[(long)j * d + c] += alpha * du * qi[c];
                dv[(long)j * d + c] += p[j] * doi[c];
            }
        }
    }
    if (dsink) *dsink = sink ? ds_sink : 0.0;
    free(s); free(t); free(p); free(dp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The tiled online algorithm, FP64, one head: the method's own steps, kept  */
/* separate from the one-pass definition above so that each pins the other. */
/*                                                                           */
/* [FA3H] sec. 4.2 / [FAv4] "common computation graph": key tiles are        */
/* processed one at a time in a caller-given order; per row the state is     */
/* (reference r, sum l, unnormalised U).  Scores are taken in base 2,        */
/* X = S * log2(e) with S = alpha * q.k (the pages fold alpha*log2 e into    */
/* one constant).  For a new tile with row max b ([FAv4] "conditional        */
/* rescale"):                                                                */
/*    r' = max(r, b)  if  max(r, b) - r > tau,   else r                      */
/*    scale = 2^(r - r');  l = scale*l + sum 2^(X - r');                     */
/*    U = scale*U + sum 2^(X - r') v                                         */
/* The first tile that has a finite maximum initialises r = b.  tau = 0 is   */
/* the plain online softmax (r is then the running maximum).  At the end     */
/* O = U / l and LSE = r ln 2 + ln l; a row that never saw a finite score    */
/* gets O = 0, LSE = -inf ([FA3H] sec. 4.6).                                 */
/*                                                                           */
/* tile_lo[t], tile_hi[t] give the key range [lo, hi) of the t-th tile in   */
/* processing order (any order, any sizes; ranges may be empty).             */
/* n_rescales (optional) returns how many (row, tile) steps moved r.        */
/* ------------------------------------------------------------------------ */
int oracle_attention_online_head(const double *q, const double *k,
                                 const double *v, int Nq, int Nk, int d,
                                 long ldq, long ldk, long ldv, double alpha,
                                 int causal, const int *tile_lo,
                                 const int *tile_hi, int n_tiles, double tau,
                                 double *o, long ldo, double *lse,
                                 long *n_rescales)
{
    if (Nq < 0 || Nk < 0 || d < 1 || n_tiles < 0) return -1;
    const double log2e = 1.4426950408889634073599246810018921;
    const double ln2 = 0.6931471805599453094172321214581766;
    double *x = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double *u = (double *)malloc(sizeof(double) * (size_t)d);
    if (!x || !u) { free(x); free(u); return -1; }
    long rescales = 0;
    for (int i = 0; i < Nq; ++i) {
        const double *qi = q + (long)i * ldq;
        double r = -INFINITY, l = 0.0;
        int started = 0;
        for (int c = 0; c < d; ++c) u[c] = 0.0;
        for (int t = 0; t < n_tiles; ++t) {
            int lo = tile_lo[t], hi = tile_hi[t];
            if (lo < 0 || hi > Nk || lo > hi) { free(x); free(u); return -1; }
            double b = -INFINITY;
            for (int j = lo; j < hi; ++j) {
                if (visible(i, j, Nq, Nk, causal)) {
                    double dot = 0.0;
                    const double *kj = k + (long)j * ldk;
                    for (int c = 0; c < d; ++c) dot += qi[c] * kj[c];
                    x[j] = alpha * dot * log2e;
                } else {
                    x[j] = -INFINITY;
                }
                if (x[j] > b) b = x[j];
            }
            if (b == -INFINITY) continue;        /* tile contributes nothing */
            double rn, scale;
            if (!started) {                      /* first tile initialises r */
                rn = b;
                scale = 1.0;                     /* l and U are still zero */
                started = 1;
            } else {
                double mx = (b > r) ? b : r;
                rn = (mx - r > tau) ? mx : r;
                scale = exp2(r - rn);
                if (rn != r) ++rescales;
            }
            l *= scale;
            for (int c = 0; c < d; ++c) u[c] *= scale;
            for (int j = lo; j < hi; ++j) {
                if (x[j] == -INFINITY) continue;
                double pj = exp2(x[j] - rn);
                l += pj;
                const double *vj = v + (long)j * ldv;
                for (int c = 0; c < d; ++c) u[c] += pj * vj[c];
            }
            r = rn;
        }
        double *oi = o + (long)i * ldo;
        if (!started || l == 0.0) {
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            lse[i] = -INFINITY;
        } else {
            for (int c = 0; c < d; ++c) oi[c] = u[c] / l;
            lse[i] = r * ln2 + log(l);
        }
    }
    if (n_rescales) *n_rescales = rescales;
    free(x);
    free(u);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Incoherent processing, [FA3H] sec. 6.4: x <- x M with                     */
/* M = (1/sqrt d) H D, H the d x d Sylvester Hadamard matrix                 */
/* (H_ik = (-1)^popcount(i & k)), D = diag(signs), signs[k] = +-1.           */
/* Written as the plain O(d^2) product, not the fast transform.              */
/* Rows of x are n_rows vectors of length d at stride ld.                    */
/* ------------------------------------------------------------------------ */
static int popcount_u32(unsigned int a)
{
    int n = 0;
    while (a) { n += (int)(a & 1u); a >>= 1; }
    return n;
}

int oracle_hadamard_rotate(const double *x, double *y, long n_rows, int d,
                           long ld, const double *signs)
{
    if (d < 1 || (d & (d - 1)) != 0 || !x || !y || !signs) return -1;
    double inv = 1.0 / sqrt((double)d);
    for (long r = 0; r < n_rows; ++r) {
        const double *xr = x + r * ld;
        double *yr = y + r * ld;
        for (int kk = 0; kk < d; ++kk) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) {
                double hik = (popcount_u32((unsigned)(i & kk)) & 1) ? -1.0 : 1.0;
                acc += xr[i] * hik;
            }
            yr[kk] = acc * inv * signs[kk];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 e4m3 ("e4m3fn": bias 7, 3 mantissa bits, no infinities, max finite    */
/* 448, 0x7f / 0xff = NaN).  [FA3H] sec. 6.1 gives the range +-448.           */
/* decode: the value a code stands for.  encode: round to nearest, ties to    */
/* even mantissa, saturating at +-448 (finite inputs only).                  */
/* ------------------------------------------------------------------------ */
double oracle_e4m3_decode(unsigned int code)
{
    unsigned int s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double val;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) val = ldexp((double)m, -9);          /* subnormal: m/8 * 2^-6 */
    else val = ldexp(8.0 + (double)m, (int)e - 10);   /* (1 + m/8) 2^(e-7) */
    return s ? -val : val;
}

unsigned int oracle_e4m3_encode(double x)
{
    if (x != x) return 0x7fu;
    unsigned int sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80u : 0u;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7eu;              /* saturate */
    /* candidates: all non-negative finite codes 0x00..0x7e are monotone in
       value; pick the nearest, ties to the even code (even mantissa). */
    unsigned int lo = 0, hi = 0x7e;
    while (hi - lo > 1) {                             /* largest code <= a */
        unsigned int mid = (lo + hi) / 2;
        if (oracle_e4m3_decode(mid) <= a) lo = mid; else hi = mid;
    }
    if (oracle_e4m3_decode(hi) <= a) lo = hi;
    if (lo == 0x7e) return sign | lo;
    double vlo = oracle_e4m3_decode(lo), vhi = oracle_e4m3_decode(lo + 1);
    double dlo = a - vlo, dhi = vhi - a;
    unsigned int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = lo + 1;
    else c = (lo & 1u) ? lo + 1 : lo;
    return sign | c;
}

/*
 * Block quantization, [FA3H] sec. 6.3: one FP32 scale per tile of
 * tile_rows rows (all d columns) of one head.  scale = amax / 448 (an
 * all-zero tile gets scale 1); code = e4m3(x / scale).  The scale is
 * rounded to float, and x / scale is evaluated in FP64 from that float.
 * x: n_rows x d at stride ld; codes written at the same positions of
 * `codes` (stride ld); scales[t] for tile t.
 */
int oracle_quantize_e4m3_tiles(const double *x, unsigned char *codes,
                               float *scales, long n_rows, int d, long ld,
                               int tile_rows)
{
    if (tile_rows < 1 || d < 1) return -1;
    long n_tiles = (n_rows + tile_rows - 1) / tile_rows;
    for (long t = 0; t < n_tiles; ++t) {
        long r0 = t * tile_rows, r1 = r0 + tile_rows;
        if (r1 > n_rows) r1 = n_rows;
        double amax = 0.0;
        for (long r = r0; r < r1; ++r)
            for (int c = 0; c < d; ++c) {
                double a = fabs(x[r * ld + c]);
                if (a > amax) amax = a;
            }
        float sc = (amax > 0.0) ? (float)(amax / 448.0) : 1.0f;
        scales[t] = sc;
        for (long r = r0; r < r1; ++r)
            for (int c = 0; c < d; ++c)
                codes[r * ld + c] =
                    (unsigned char)oracle_e4m3_encode(x[r * ld + c] / (double)sc);
    }
    return 0;
}
