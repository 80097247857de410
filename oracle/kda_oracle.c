/*
 * kda_oracle.c -- plain fp64 CPU oracle for the Kimi Delta Attention (KDA)
 * forward prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the CUDA
 * path: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA
 * library, and it never reads a value produced by that library.
 *
 * What it computes (the definition, per sequence n and head h, t = 1..L_n):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * with S in R^{Dk x Dv}, S_0 = initial state (or zero) and final = S_{L_n}.
 * Source: Kimi Delta Attention, the gated delta rule with a per-channel decay
 * gate (the pages name the method but print no formula); the pages
 * ("feat(kda/sm90): FlashKDA prefill port + intracard-CP prefill", commit
 * notes) fix chunks of 16 tokens, head size 128 and the forward pass only;
 * they split the work into K1 (decayed q/k, beta and the WY inverse per chunk)
 * and K2 (the state carried from chunk to chunk), and the segment pipeline into
 * K1 once, per-segment summaries (pre_scan), the merge, and K2 per segment.
 *
 * Three independent forms are provided:
 *   kda_oracle_recurrent  token by token, the formula written out (O1).
 *   kda_oracle_chunked    the chunkwise (WY) form derived from O1 (O2).
 *   kda_oracle_segmented  the segment form: per-segment summaries
 *                         (transition m_seg, offset b_seg), a serial merge of
 *                         carries, then the chunked pass per segment.
 *
 * Layouts (row-major, all fp64): q,k,g: [T_total][H][Dk]; v,out: [T_total][H][Dv];
 * beta: [T_total][H]; states: [N][H][Dk][Dv] indexed [n][h][i_k][j_v].
 * Sequences are given by cu[0..N] (cu[0] = 0, non-decreasing, cu[N] = T_total).
 * A NULL initial state means zero; a NULL final-state pointer means "not written".
 *
 * Return value: 0 on success, -1 on invalid arguments, -2 on allocation failure.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const double *s0;
    double *out, *sfin;
    const int64_t *cu;
    int64_t n_seqs, H, Dk, Dv;
    double scale;
} problem;

static int check_problem(const problem *p) {
    if (p->n_seqs < 0 || p->H <= 0 || p->Dk <= 0 || p->Dv <= 0) return -1;
    if (!p->cu) return -1;
    if (p->cu[0] != 0) return -1;
    for (int64_t n = 0; n < p->n_seqs; ++n)
        if (p->cu[n + 1] < p->cu[n]) return -1;
    if (p->cu[p->n_seqs] > 0 && (!p->q || !p->k || !p->v || !p->g || !p->beta || !p->out))
        return -1;
    return 0;
}

static void load_state(const problem *p, int64_t n, int64_t h, double *S) {
    const size_t sz = (size_t)(p->Dk * p->Dv);
    if (p->s0)
        memcpy(S, p->s0 + ((size_t)n * p->H + h) * sz, sz * sizeof(double));
    else
        memset(S, 0, sz * sizeof(double));
}

static void store_state(const problem *p, int64_t n, int64_t h, const double *S) {
    const size_t sz = (size_t)(p->Dk * p->Dv);
    if (p->sfin) memcpy(p->sfin + ((size_t)n * p->H + h) * sz, S, sz * sizeof(double));
}

/* ---------------------------------------------------------------------------
 * O1: the recurrence, one token at a time.
 *   P   = Diag(exp g_t) S_{t-1}            (decay first)
 *   u   = P^T k_t                           (current prediction for key k_t)
 *   S_t = P + k_t (beta_t (v_t - u))^T      (= (I - b k k^T) P + b k v^T)
 *   o_t = scale S_t^T q_t
 * ------------------------------------------------------------------------- */
static void recurrent_chain(const problem *p, int64_t n, int64_t h, double *S, double *u) {
    const int64_t H = p->H, Dk = p->Dk, Dv = p->Dv;
    load_state(p, n, h, S);
    for (int64_t t = p->cu[n]; t < p->cu[n + 1]; ++t) {
        const double *qt = p->q + ((size_t)t * H + h) * Dk;
        const double *kt = p->k + ((size_t)t * H + h) * Dk;
        const double *gt = p->g + ((size_t)t * H + h) * Dk;
        const double *vt = p->v + ((size_t)t * H + h) * Dv;
        const double bt = p->beta[(size_t)t * H + h];
        double *ot = p->out + ((size_t)t * H + h) * Dv;
        for (int64_t i = 0; i < Dk; ++i) {
            const double d = exp(gt[i]);
            for (int64_t j = 0; j < Dv; ++j) S[i * Dv + j] *= d;
        }
        for (int64_t j = 0; j < Dv; ++j) u[j] = 0.0;
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t j = 0; j < Dv; ++j) u[j] += S[i * Dv + j] * kt[i];
        for (int64_t j = 0; j < Dv; ++j) u[j] = bt * (vt[j] - u[j]);
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t j = 0; j < Dv; ++j) S[i * Dv + j] += kt[i] * u[j];
        for (int64_t j = 0; j < Dv; ++j) ot[j] = 0.0;
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t j = 0; j < Dv; ++j) ot[j] += S[i * Dv + j] * qt[i];
        for (int64_t j = 0; j < Dv; ++j) ot[j] *= p->scale;
    }
    store_state(p, n, h, S);
}

/* ---------------------------------------------------------------------------
 * O2: the chunkwise form.  For one chunk of C rows starting at token t0 with
 * chunk-start state S (all sums over the chunk's rows, 0-based r, s):
 *   gam[r]   = sum_{m<=r} g[m]                        (in-chunk cumulative, per channel)
 *   A[r][s]  = beta_r sum_i k_r[i] k_s[i] exp(gam_r[i]-gam_s[i])       (s < r)
 *   T        = (I + A)^{-1}                            (unit lower triangular)
 *   W        = T diag(beta) Ktil,  Ktil[s][i] = k_s[i] exp(gam_s[i])
 *   U        = T diag(beta) V
 *   delta    = U - W S
 *   O        = scale (Qtil S + Mq delta),  Qtil[r][i] = q_r[i] exp(gam_r[i]),
 *              Mq[r][s] = sum_i q_r[i] k_s[i] exp(gam_r[i]-gam_s[i])  (s <= r)
 *   S_next   = Diag(exp gam_last) S + sum_s Kbar_s delta_s^T,
 *              Kbar_s[i] = k_s[i] exp(gam_last[i] - gam_s[i])
 * Derivation: unroll S_r = Diag(exp g_r) S_{r-1} + k_r delta_r^T with
 * delta_r = beta_r (v_r - (Diag(exp g_r) S_{r-1})^T k_r) inside the chunk; the
 * rows of delta then satisfy (I + A) delta = diag(beta) (V - Ktil S).
 * ------------------------------------------------------------------------- */
typedef struct {
    double *gam, *A, *T, *W, *U, *delta, *Mq, *Snew;
} chunk_ws;

static int chunk_ws_alloc(chunk_ws *w, int64_t C, int64_t Dk, int64_t Dv) {
    w->gam = malloc(sizeof(double) * C * Dk);
    w->A = malloc(sizeof(double) * C * C);
    w->T = malloc(sizeof(double) * C * C);
    w->W = malloc(sizeof(double) * C * Dk);
    w->U = malloc(sizeof(double) * C * Dv);
    w->delta = malloc(sizeof(double) * C * Dv);
    w->Mq = malloc(sizeof(double) * C * C);
    w->Snew = malloc(sizeof(double) * Dk * Dv);
    return (w->gam && w->A && w->T && w->W && w->U && w->delta && w->Mq && w->Snew) ? 0 : -2;
}

static void chunk_ws_free(chunk_ws *w) {
    free(w->gam); free(w->A); free(w->T); free(w->W);
    free(w->U); free(w->delta); free(w->Mq); free(w->Snew);
}

/* Chunk quantities that do not depend on the state: gam, A, T, W, U, Mq. */
static void chunk_prepare(const problem *p, int64_t h, int64_t t0, int64_t C, chunk_ws *w) {
    const int64_t H = p->H, Dk = p->Dk, Dv = p->Dv;
#define KROW(r) (p->k + ((size_t)(t0 + (r)) * H + h) * Dk)
#define QROW(r) (p->q + ((size_t)(t0 + (r)) * H + h) * Dk)
#define GROW(r) (p->g + ((size_t)(t0 + (r)) * H + h) * Dk)
#define VROW(r) (p->v + ((size_t)(t0 + (r)) * H + h) * Dv)
#define BETA(r) (p->beta[(size_t)(t0 + (r)) * H + h])
    for (int64_t i = 0; i < Dk; ++i) {
        double acc = 0.0;
        for (int64_t r = 0; r < C; ++r) {
            acc += GROW(r)[i];
            w->gam[r * Dk + i] = acc;
        }
    }
    for (int64_t r = 0; r < C; ++r)
        for (int64_t s = 0; s < C; ++s) {
            double a = 0.0, m = 0.0;
            if (s <= r) {
                for (int64_t i = 0; i < Dk; ++i) {
                    const double e = exp(w->gam[r * Dk + i] - w->gam[s * Dk + i]);
                    a += KROW(r)[i] * KROW(s)[i] * e;
                    m += QROW(r)[i] * KROW(s)[i] * e;
                }
            }
            w->A[r * C + s] = (s < r) ? BETA(r) * a : 0.0;
            w->Mq[r * C + s] = (s <= r) ? m : 0.0;
        }
    /* Forward substitution for T = (I + A)^{-1}: column s of T solves
       (I + A) x = e_s, so x_r = [r == s] - sum_{s <= m < r} A[r][m] x_m. */
    for (int64_t s = 0; s < C; ++s)
        for (int64_t r = 0; r < C; ++r) {
            double x = (r == s) ? 1.0 : 0.0;
            if (r > s)
                for (int64_t m = s; m < r; ++m) x -= w->A[r * C + m] * w->T[m * C + s];
            w->T[r * C + s] = (r >= s) ? x : 0.0;
        }
    for (int64_t r = 0; r < C; ++r) {
        for (int64_t i = 0; i < Dk; ++i) {
            double acc = 0.0;
            for (int64_t s = 0; s <= r; ++s)
                acc += w->T[r * C + s] * BETA(s) * KROW(s)[i] * exp(w->gam[s * Dk + i]);
            w->W[r * Dk + i] = acc;
        }
        for (int64_t j = 0; j < Dv; ++j) {
            double acc = 0.0;
            for (int64_t s = 0; s <= r; ++s) acc += w->T[r * C + s] * BETA(s) * VROW(s)[j];
            w->U[r * Dv + j] = acc;
        }
    }
}

/* Run one chunk from state S (updated in place); writes outputs if out_rows. */
static void chunk_step(const problem *p, int64_t h, int64_t t0, int64_t C, chunk_ws *w,
                       double *S, int write_out) {
    const int64_t H = p->H, Dk = p->Dk, Dv = p->Dv;
    chunk_prepare(p, h, t0, C, w);
    for (int64_t r = 0; r < C; ++r)
        for (int64_t j = 0; j < Dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < Dk; ++i) acc += w->W[r * Dk + i] * S[i * Dv + j];
            w->delta[r * Dv + j] = w->U[r * Dv + j] - acc;
        }
    if (write_out)
        for (int64_t r = 0; r < C; ++r) {
            double *orow = p->out + ((size_t)(t0 + r) * H + h) * Dv;
            for (int64_t j = 0; j < Dv; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < Dk; ++i)
                    acc += QROW(r)[i] * exp(w->gam[r * Dk + i]) * S[i * Dv + j];
                for (int64_t s = 0; s <= r; ++s) acc += w->Mq[r * C + s] * w->delta[s * Dv + j];
                orow[j] = p->scale * acc;
            }
        }
    const double *glast = w->gam + (C - 1) * Dk;
    for (int64_t i = 0; i < Dk; ++i) {
        const double d = exp(glast[i]);
        for (int64_t j = 0; j < Dv; ++j) {
            double acc = d * S[i * Dv + j];
            for (int64_t s = 0; s < C; ++s)
                acc += KROW(s)[i] * exp(glast[i] - w->gam[s * Dk + i]) * w->delta[s * Dv + j];
            w->Snew[i * Dv + j] = acc;
        }
    }
    memcpy(S, w->Snew, sizeof(double) * Dk * Dv);
}

static int chunked_chain(const problem *p, int64_t n, int64_t h, int64_t C, double *S) {
    chunk_ws w;
    if (chunk_ws_alloc(&w, C, p->Dk, p->Dv)) { chunk_ws_free(&w); return -2; }
    load_state(p, n, h, S);
    for (int64_t t0 = p->cu[n]; t0 < p->cu[n + 1]; t0 += C) {
        const int64_t rows = (p->cu[n + 1] - t0 < C) ? p->cu[n + 1] - t0 : C;
        chunk_step(p, h, t0, rows, &w, S, 1);
    }
    store_state(p, n, h, S);
    chunk_ws_free(&w);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Segment form.  Over one chunk the state map is affine:
 *   S_next = Acal S + b,   Acal = Diag(exp gam_last) - Kbar^T W,   b = Kbar^T U
 * (substitute delta = U - W S into the S_next line above).  For a segment of
 * chunks: m_seg = product of the chunk transitions (latest on the left) and
 * b_seg = the state reached from zero ("pre_scan").  The carries follow
 *   carry_0 = S_0,  carry_{s+1} = m_seg[s] carry_s + b_seg[s]    ("merge"),
 * and each segment is then run from its carry with outputs ("segment-K2").
 * Segments are seg_len tokens long (a multiple of the chunk length) from each
 * sequence's start; the last one may be shorter.
 * ------------------------------------------------------------------------- */
static int segmented_chain(const problem *p, int64_t n, int64_t h, int64_t C, int64_t seg_len,
                           double *S) {
    const int64_t Dk = p->Dk, Dv = p->Dv;
    const int64_t L = p->cu[n + 1] - p->cu[n];
    const int64_t nseg = (L + seg_len - 1) / seg_len;
    chunk_ws w;
    int rc = chunk_ws_alloc(&w, C, Dk, Dv);
    double *m_seg = malloc(sizeof(double) * (nseg ? nseg : 1) * Dk * Dk);
    double *b_seg = malloc(sizeof(double) * (nseg ? nseg : 1) * Dk * Dv);
    double *Acal = malloc(sizeof(double) * Dk * Dk);
    double *tmpm = malloc(sizeof(double) * Dk * Dk);
    double *tmpb = malloc(sizeof(double) * Dk * Dv);
    double *carry = malloc(sizeof(double) * Dk * Dv);
    if (rc || !m_seg || !b_seg || !Acal || !tmpm || !tmpb || !carry) { rc = -2; goto done; }

    /* pre_scan: per-segment transition and offset (the last segment needs none). */
    for (int64_t sg = 0; sg + 1 < nseg; ++sg) {
        double *M = m_seg + sg * Dk * Dk, *B = b_seg + sg * Dk * Dv;
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t i2 = 0; i2 < Dk; ++i2) M[i * Dk + i2] = (i == i2) ? 1.0 : 0.0;
        memset(B, 0, sizeof(double) * Dk * Dv);
        const int64_t s_begin = p->cu[n] + sg * seg_len;
        const int64_t s_end = (s_begin + seg_len < p->cu[n + 1]) ? s_begin + seg_len : p->cu[n + 1];
        for (int64_t t0 = s_begin; t0 < s_end; t0 += C) {
            const int64_t rows = (s_end - t0 < C) ? s_end - t0 : C;
            chunk_prepare(p, h, t0, rows, &w);
            const double *glast = w.gam + (rows - 1) * Dk;
            /* Acal = Diag(exp glast) - Kbar^T W ; b = Kbar^T U */
            for (int64_t i = 0; i < Dk; ++i) {
                for (int64_t i2 = 0; i2 < Dk; ++i2) {
                    double acc = (i == i2) ? exp(glast[i]) : 0.0;
                    for (int64_t s = 0; s < rows; ++s)
                        acc -= p->k[((size_t)(t0 + s) * p->H + h) * Dk + i] *
                               exp(glast[i] - w.gam[s * Dk + i]) * w.W[s * Dk + i2];
                    Acal[i * Dk + i2] = acc;
                }
            }
            for (int64_t i = 0; i < Dk; ++i)
                for (int64_t j = 0; j < Dv; ++j) {
                    double acc = 0.0;
                    for (int64_t i2 = 0; i2 < Dk; ++i2) acc += Acal[i * Dk + i2] * B[i2 * Dv + j];
                    for (int64_t s = 0; s < rows; ++s)
                        acc += p->k[((size_t)(t0 + s) * p->H + h) * Dk + i] *
                               exp(glast[i] - w.gam[s * Dk + i]) * w.U[s * Dv + j];
                    tmpb[i * Dv + j] = acc;
                }
            memcpy(B, tmpb, sizeof(double) * Dk * Dv);
            for (int64_t i = 0; i < Dk; ++i)
                for (int64_t i2 = 0; i2 < Dk; ++i2) {
                    double acc = 0.0;
                    for (int64_t m = 0; m < Dk; ++m) acc += Acal[i * Dk + m] * M[m * Dk + i2];
                    tmpm[i * Dk + i2] = acc;
                }
            memcpy(M, tmpm, sizeof(double) * Dk * Dk);
        }
    }
    /* merge + segment-K2 */
    load_state(p, n, h, carry);
    for (int64_t sg = 0; sg < nseg; ++sg) {
        memcpy(S, carry, sizeof(double) * Dk * Dv);
        const int64_t s_begin = p->cu[n] + sg * seg_len;
        const int64_t s_end = (s_begin + seg_len < p->cu[n + 1]) ? s_begin + seg_len : p->cu[n + 1];
        for (int64_t t0 = s_begin; t0 < s_end; t0 += C) {
            const int64_t rows = (s_end - t0 < C) ? s_end - t0 : C;
            chunk_step(p, h, t0, rows, &w, S, 1);
        }
        if (sg + 1 == nseg) break;
        const double *M = m_seg + sg * Dk * Dk, *B = b_seg + sg * Dk * Dv;
        for (int64_t i = 0; i < Dk; ++i)
            for (int64_t j = 0; j < Dv; ++j) {
                double acc = B[i * Dv + j];
                for (int64_t m = 0; m < Dk; ++m) acc += M[i * Dk + m] * carry[m * Dv + j];
                tmpb[i * Dv + j] = acc;
            }
        memcpy(carry, tmpb, sizeof(double) * Dk * Dv);
    }
    /* The last segment-K2 pass ends at the final state (S0 for an empty sequence). */
    if (nseg == 0) memcpy(S, carry, sizeof(double) * Dk * Dv);
    store_state(p, n, h, S);
done:
    chunk_ws_free(&w);
    free(m_seg); free(b_seg); free(Acal); free(tmpm); free(tmpb); free(carry);
    return rc;
}

/* ------------------------------------------------------------------------- */
enum { FORM_RECURRENT = 0, FORM_CHUNKED = 1, FORM_SEGMENTED = 2 };

static int run_all(const problem *p, int form, int64_t C, int64_t seg_len, int n_threads) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (form != FORM_RECURRENT && C <= 0) return -1;
    if (form == FORM_SEGMENTED && (seg_len <= 0 || seg_len % C)) return -1;
    const int64_t units = p->n_seqs * p->H;
    int err = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel reduction(min : err)
    {
        double *S = malloc(sizeof(double) * p->Dk * p->Dv);
        double *u = malloc(sizeof(double) * p->Dv);
        if (!S || !u) err = -2;
#pragma omp for schedule(dynamic, 1)
        for (int64_t unit = 0; unit < units; ++unit) {
            if (!S || !u) continue;
            const int64_t n = unit / p->H, h = unit % p->H;
            int e = 0;
            if (form == FORM_RECURRENT) recurrent_chain(p, n, h, S, u);
            else if (form == FORM_CHUNKED) e = chunked_chain(p, n, h, C, S);
            else e = segmented_chain(p, n, h, C, seg_len, S);
            if (e < err) err = e;
        }
        free(S);
        free(u);
    }
    return err;
}

#define PROBLEM_INIT                                                                     \
    problem p = {q, k, v, g, beta, s0, out, sfin, cu, n_seqs, H, Dk, Dv, scale};

int kda_oracle_recurrent(int64_t n_seqs, const int64_t *cu, int64_t H, int64_t Dk, int64_t Dv,
                         const double *q, const double *k, const double *v, const double *g,
                         const double *beta, double scale, const double *s0, double *out,
                         double *sfin, int n_threads) {
    PROBLEM_INIT
    return run_all(&p, FORM_RECURRENT, 0, 0, n_threads);
}

int kda_oracle_chunked(int64_t n_seqs, const int64_t *cu, int64_t H, int64_t Dk, int64_t Dv,
                       const double *q, const double *k, const double *v, const double *g,
                       const double *beta, double scale, const double *s0, double *out,
                       double *sfin, int64_t chunk, int n_threads) {
    PROBLEM_INIT
    return run_all(&p, FORM_CHUNKED, chunk, 0, n_threads);
}

int kda_oracle_segmented(int64_t n_seqs, const int64_t *cu, int64_t H, int64_t Dk, int64_t Dv,
                         const double *q, const double *k, const double *v, const double *g,
                         const double *beta, double scale, const double *s0, double *out,
                         double *sfin, int64_t chunk, int64_t seg_len, int n_threads) {
    PROBLEM_INIT
    return run_all(&p, FORM_SEGMENTED, chunk, seg_len, n_threads);
}

int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
