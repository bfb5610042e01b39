/*
 * oracle.c -- plain, slow, fp64 CPU oracle for striped causal attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code with the CUDA library.
 *
 * What it computes (sources are the pages on "Striped Attention: Faster Ring
 * Attention for Causal Transformers"):
 *  - Exact causal softmax attention on the UNPERMUTED sequence.  The summary
 *    page (research.elamur.ai, §Summary) and the abstract (pith.science paper
 *    page, abstract) state that Ring/Striped Attention are exact attention
 *    algorithms and that the striped permutation leaves the output exact
 *    (attention is permutation-equivariant; §Key points "Striped layout").
 *    So the definition the GPU path must reach is plain causal attention:
 *        s_pt  = scale * <q_p, k_t>            for t <= p
 *        LSE_p = log sum_{t<=p} exp(s_pt)      (natural log)
 *        P_pt  = exp(s_pt - LSE_p)
 *        O_p   = sum_{t<=p} P_pt v_t
 *  - The backward pass by direct differentiation of that definition (the
 *    pages say the method is used for training, §Summary; they give no
 *    formulas).  With dO the output cotangent:
 *        dP_pt = <dO_p, v_t>
 *        J_p   = sum_t P_pt dP_pt              (softmax Jacobian row sum)
 *        dS_pt = P_pt (dP_pt - J_p)
 *        dQ_p  = scale * sum_t dS_pt k_t
 *        dK_t  = scale * sum_{p>=t} dS_pt q_p
 *        dV_t  = sum_{p>=t} P_pt dO_p
 *  - The stripe placement: "every N-th token" (§Summary) -- virtual device d
 *    holds global positions p with p mod N == d, in increasing order, so
 *    stripe-major row d*L + i holds position i*N + d (L = S/N).  The
 *    contiguous (Ring Attention) placement gives device d positions
 *    [d*L, (d+1)*L) (§Summary, first paragraph).
 *  - A third placement that the pages do not describe, kept for comparison
 *    with the striped one: the zig-zag (load-balanced) placement cuts the
 *    sequence into 2N chunks of C = S/(2N) positions and gives device d
 *    chunk d followed by chunk 2N-1-d (one chunk from each end), so row
 *    d*L + i holds d*C + i for i < C and (2N-1-d)*C + (i - C) otherwise.
 *  - Per-round work: in round r device d holds the key/value stripe of
 *    device e = (d - r) mod N (key/value blocks circulate around the ring,
 *    §Summary).  A Tq x Tk tile of (query, key) pairs of that round is
 *    counted when at least one of its pairs is kept by global causality;
 *    it is "full" when every pair in it is kept, "partial" otherwise.  The
 *    brute-force counter below enumerates every pair; the closed forms are
 *    the algebra of the same definition for tiles that divide L.
 *
 * Everything is fp64.  Rows are split across POSIX threads; there is no
 * blocking, fusion or reordering of the arithmetic beyond the definitions.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Thread pool helper: run fn(arg, lo, hi) over [0, n) split in nthreads.   */
/* ------------------------------------------------------------------------ */
typedef void (*range_fn)(void *arg, int64_t lo, int64_t hi);

typedef struct {
    range_fn fn;
    void *arg;
    int64_t n;
    int64_t chunk;
    int64_t *next; /* shared cursor */
    pthread_mutex_t *mu;
} worker_t;

static void *worker_main(void *p) {
    worker_t *w = (worker_t *)p;
    for (;;) {
        int64_t lo;
        pthread_mutex_lock(w->mu);
        lo = *w->next;
        *w->next += w->chunk;
        pthread_mutex_unlock(w->mu);
        if (lo >= w->n) break;
        int64_t hi = lo + w->chunk;
        if (hi > w->n) hi = w->n;
        w->fn(w->arg, lo, hi);
    }
    return NULL;
}

static void parallel_for(range_fn fn, void *arg, int64_t n, int nthreads, int64_t chunk) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (chunk < 1) chunk = 1;
    if (nthreads == 1) {
        fn(arg, 0, n);
        return;
    }
    int64_t next = 0;
    pthread_mutex_t mu;
    pthread_mutex_init(&mu, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    worker_t w = {fn, arg, n, chunk, &next, &mu};
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker_main, &w);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&mu);
}

static double dot(const double *a, const double *b, int64_t D) {
    double s = 0.0;
    for (int64_t c = 0; c < D; ++c) s += a[c] * b[c];
    return s;
}

/* ------------------------------------------------------------------------ */
/* Stripe placement                                                         */
/* ------------------------------------------------------------------------ */

/* Global position held by row `row` of the layout.
 * layout 0 = striped: row d*L + i holds position i*N + d.
 * layout 1 = contiguous: row r holds position r.
 * layout 2 = zig-zag: row d*L + i holds d*C + i (i < C) or
 *            (2N-1-d)*C + (i - C) (i >= C), C = S/(2N).                    */
int64_t oracle_position_of_row(int64_t row, int64_t S, int N, int layout) {
    if (layout == 1) return row;
    int64_t L = S / N;
    int64_t d = row / L, i = row % L;
    if (layout == 2) {
        int64_t C = S / (2 * (int64_t)N);
        return i < C ? d * C + i : (2 * (int64_t)N - 1 - d) * C + (i - C);
    }
    return i * (int64_t)N + d;
}

/* Fill pos[row] for every row, by enumerating positions: device d collects,
 * in increasing order, every position p with p mod N == d. */
void oracle_stripe_positions(int64_t S, int N, int64_t *pos) {
    int64_t row = 0;
    for (int d = 0; d < N; ++d)
        for (int64_t p = 0; p < S; ++p)
            if (p % N == d) pos[row++] = p;
}

/* Fill pos[row] for the zig-zag placement, by enumerating positions: device
 * d collects, in increasing order, every position whose chunk index p / C
 * is d or 2N-1-d (C = S/(2N), S divisible by 2N). */
void oracle_zigzag_positions(int64_t S, int N, int64_t *pos) {
    int64_t C = S / (2 * (int64_t)N), row = 0;
    for (int d = 0; d < N; ++d)
        for (int64_t p = 0; p < S; ++p) {
            int64_t chunk = p / C;
            if (chunk == d || chunk == 2 * (int64_t)N - 1 - d) pos[row++] = p;
        }
}

/* ------------------------------------------------------------------------ */
/* Forward: one head, selected query rows, optional key subset              */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v;
    int64_t S, D;
    double scale;
    const int64_t *rows; /* query positions (NULL: all) */
    const unsigned char *key_in_set; /* NULL: every key */
    double *o, *lse;     /* outputs indexed by slot in rows[] */
} fwd_args;

static void fwd_range(void *vp, int64_t lo, int64_t hi) {
    fwd_args *a = (fwd_args *)vp;
    const int64_t D = a->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)a->S);
    for (int64_t idx = lo; idx < hi; ++idx) {
        int64_t p = a->rows ? a->rows[idx] : idx;
        const double *qp = a->q + p * D;
        /* scores for kept keys t <= p (and in the key set) */
        double m = -INFINITY;
        int64_t kept = 0;
        for (int64_t t = 0; t <= p; ++t) {
            if (a->key_in_set && !a->key_in_set[t]) continue;
            s[t] = a->scale * dot(qp, a->k + t * D, D);
            if (s[t] > m) m = s[t];
            ++kept;
        }
        double *op = a->o + idx * D;
        for (int64_t c = 0; c < D; ++c) op[c] = 0.0;
        if (kept == 0) { /* empty key set: zero output, LSE = -inf */
            a->lse[idx] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int64_t t = 0; t <= p; ++t) {
            if (a->key_in_set && !a->key_in_set[t]) continue;
            sum += exp(s[t] - m);
        }
        double lse = m + log(sum);
        a->lse[idx] = lse;
        for (int64_t t = 0; t <= p; ++t) {
            if (a->key_in_set && !a->key_in_set[t]) continue;
            double P = exp(s[t] - lse);
            const double *vt = a->v + t * D;
            for (int64_t c = 0; c < D; ++c) op[c] += P * vt[c];
        }
    }
    free(s);
}

/* O and LSE for query positions rows[0..nrows) (all S rows when rows is
 * NULL) of one head stored [S, D] row-major in position order.  When
 * key_in_set is non-NULL only keys t with key_in_set[t] != 0 take part
 * (the per-round partial result of one ring round); a row with no kept key
 * gets O = 0 and LSE = -inf. */
void oracle_attn_fwd(const double *q, const double *k, const double *v, int64_t S, int64_t D,
                     double scale, const int64_t *rows, int64_t nrows,
                     const unsigned char *key_in_set, double *o, double *lse, int nthreads) {
    fwd_args a = {q, k, v, S, D, scale, rows, key_in_set, o, lse};
    int64_t n = rows ? nrows : S;
    parallel_for(fwd_range, &a, n, nthreads, 16);
}

/* ------------------------------------------------------------------------ */
/* Backward                                                                 */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v, *dO;
    int64_t S, D;
    double scale;
    const int64_t *rows;
    double *lse, *J, *dq; /* per slot; dq may be NULL */
} rowstat_args;

static void rowstat_range(void *vp, int64_t lo, int64_t hi) {
    rowstat_args *a = (rowstat_args *)vp;
    const int64_t D = a->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)a->S);
    for (int64_t idx = lo; idx < hi; ++idx) {
        int64_t p = a->rows ? a->rows[idx] : idx;
        const double *qp = a->q + p * D;
        const double *dop = a->dO + p * D;
        double m = -INFINITY;
        for (int64_t t = 0; t <= p; ++t) {
            s[t] = a->scale * dot(qp, a->k + t * D, D);
            if (s[t] > m) m = s[t];
        }
        double sum = 0.0;
        for (int64_t t = 0; t <= p; ++t) sum += exp(s[t] - m);
        double lse = m + log(sum);
        /* J_p = sum_t P_pt dP_pt with dP_pt = <dO_p, v_t> */
        double J = 0.0;
        for (int64_t t = 0; t <= p; ++t) J += exp(s[t] - lse) * dot(dop, a->v + t * D, D);
        a->lse[idx] = lse;
        a->J[idx] = J;
        if (a->dq) {
            double *dqp = a->dq + idx * D;
            for (int64_t c = 0; c < D; ++c) dqp[c] = 0.0;
            for (int64_t t = 0; t <= p; ++t) {
                double P = exp(s[t] - lse);
                double dP = dot(dop, a->v + t * D, D);
                double dS = P * (dP - J);
                const double *kt = a->k + t * D;
                for (int64_t c = 0; c < D; ++c) dqp[c] += a->scale * dS * kt[c];
            }
        }
    }
    free(s);
}

/* Per-query-row quantities of the backward pass: LSE_p, J_p and (when dq is
 * non-NULL) dQ_p, for query positions rows[0..nrows) (all rows when NULL). */
void oracle_bwd_rows(const double *q, const double *k, const double *v, const double *dO,
                     int64_t S, int64_t D, double scale, const int64_t *rows, int64_t nrows,
                     double *lse, double *J, double *dq, int nthreads) {
    rowstat_args a = {q, k, v, dO, S, D, scale, rows, lse, J, dq};
    int64_t n = rows ? nrows : S;
    parallel_for(rowstat_range, &a, n, nthreads, 8);
}

typedef struct {
    const double *q, *k, *v, *dO;
    int64_t S, D;
    double scale;
    const double *lse, *J; /* indexed by p - p_lo */
    int64_t p_lo;
    const int64_t *keys;
    double *dk, *dv;
} keygrad_args;

static void keygrad_range(void *vp, int64_t lo, int64_t hi) {
    keygrad_args *a = (keygrad_args *)vp;
    const int64_t D = a->D;
    for (int64_t idx = lo; idx < hi; ++idx) {
        int64_t t = a->keys ? a->keys[idx] : idx;
        const double *kt = a->k + t * D;
        const double *vt = a->v + t * D;
        double *dkt = a->dk + idx * D;
        double *dvt = a->dv + idx * D;
        for (int64_t c = 0; c < D; ++c) dkt[c] = dvt[c] = 0.0;
        for (int64_t p = t; p < a->S; ++p) {
            const double *qp = a->q + p * D;
            const double *dop = a->dO + p * D;
            double s = a->scale * dot(qp, kt, D);
            double P = exp(s - a->lse[p - a->p_lo]);
            double dP = dot(dop, vt, D);
            double dS = P * (dP - a->J[p - a->p_lo]);
            for (int64_t c = 0; c < D; ++c) {
                dkt[c] += a->scale * dS * qp[c];
                dvt[c] += P * dop[c];
            }
        }
    }
}

/* dK_t and dV_t for key positions keys[0..nkeys) (all keys when NULL).
 * lse[] and J[] hold LSE_p and J_p for every query p in [p_lo, S); every
 * requested key must satisfy t >= p_lo. */
void oracle_bwd_keys(const double *q, const double *k, const double *v, const double *dO,
                     int64_t S, int64_t D, double scale, const double *lse, const double *J,
                     int64_t p_lo, const int64_t *keys, int64_t nkeys, double *dk, double *dv,
                     int nthreads) {
    keygrad_args a = {q, k, v, dO, S, D, scale, lse, J, p_lo, keys, dk, dv};
    int64_t n = keys ? nkeys : S;
    parallel_for(keygrad_range, &a, n, nthreads, 8);
}

/* Full backward of one head: dq, dk, dv [S, D]. */
void oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dO,
                     int64_t S, int64_t D, double scale, double *dq, double *dk, double *dv,
                     int nthreads) {
    double *lse = (double *)malloc(sizeof(double) * (size_t)S);
    double *J = (double *)malloc(sizeof(double) * (size_t)S);
    oracle_bwd_rows(q, k, v, dO, S, D, scale, NULL, S, lse, J, dq, nthreads);
    oracle_bwd_keys(q, k, v, dO, S, D, scale, lse, J, 0, NULL, S, dk, dv, nthreads);
    free(lse);
    free(J);
}

/* One ring round's share of the gradients (research.elamur.ai summary page,
 * §Summary: key/value blocks circulate and each device accumulates the work
 * of the block it holds).  The round's query rows q, dO [nq, D] sit at
 * positions qpos[], its key rows k, v [nk, D] at kpos[]; a pair takes part
 * iff kpos[t] <= qpos[p].  lse[p] and J[p] are the query rows' values over
 * the WHOLE sequence (a round sees only its own keys, the softmax of a row
 * spans them all).  Writes the round's partial dq [nq, D] (summed over the
 * round's keys) and dk, dv [nk, D] (summed over the round's queries):
 *   P_pt = exp(scale <q_p, k_t> - lse_p),  dS_pt = P_pt (<dO_p, v_t> - J_p),
 *   dq_p = scale sum_t dS_pt k_t,  dk_t = scale sum_p dS_pt q_p,
 *   dv_t = sum_p P_pt dO_p.                                               */
void oracle_bwd_block(const double *q, const double *dO, const int64_t *qpos, const double *lse,
                      const double *J, int64_t nq, const double *k, const double *v, const int64_t *kpos,
                      int64_t nk, int64_t D, double scale, double *dq, double *dk, double *dv) {
    for (int64_t i = 0; i < nq * D; ++i) dq[i] = 0.0;
    for (int64_t i = 0; i < nk * D; ++i) dk[i] = dv[i] = 0.0;
    for (int64_t p = 0; p < nq; ++p) {
        const double *qp = q + p * D, *dop = dO + p * D;
        for (int64_t t = 0; t < nk; ++t) {
            if (kpos[t] > qpos[p]) continue;
            const double *kt = k + t * D, *vt = v + t * D;
            const double P = exp(scale * dot(qp, kt, D) - lse[p]);
            const double dS = P * (dot(dop, vt, D) - J[p]);
            for (int64_t c = 0; c < D; ++c) {
                dq[p * D + c] += scale * dS * kt[c];
                dk[t * D + c] += scale * dS * qp[c];
                dv[t * D + c] += P * dop[c];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Per-round tile accounting                                                */
/* ------------------------------------------------------------------------ */

/* Brute force.  For every round r and device d (e = (d - r) mod N), every
 * query tile of Tq local rows and key tile of Tk local rows of the L x L
 * block (last tiles ragged when Tq or Tk does not divide L), enumerate all
 * pairs and keep those with key position <= query position under the
 * layout's placement.  full[r*N + d] / partial[r*N + d] receive the number
 * of tiles whose pairs are all / some-but-not-all kept.  Per (b, h).     */
void oracle_tile_counts_bruteforce(int64_t S, int N, int64_t Tq, int64_t Tk, int layout,
                                   int64_t *full, int64_t *partial) {
    int64_t L = S / N;
    for (int r = 0; r < N; ++r) {
        for (int d = 0; d < N; ++d) {
            int e = ((d - r) % N + N) % N;
            int64_t nf = 0, np = 0;
            for (int64_t i0 = 0; i0 < L; i0 += Tq) {
                int64_t i1 = i0 + Tq < L ? i0 + Tq : L;
                for (int64_t j0 = 0; j0 < L; j0 += Tk) {
                    int64_t j1 = j0 + Tk < L ? j0 + Tk : L;
                    int64_t kept = 0, total = 0;
                    for (int64_t i = i0; i < i1; ++i) {
                        int64_t p = oracle_position_of_row((int64_t)d * L + i, S, N, layout);
                        for (int64_t j = j0; j < j1; ++j) {
                            int64_t t = oracle_position_of_row((int64_t)e * L + j, S, N, layout);
                            kept += (t <= p);
                            ++total;
                        }
                    }
                    if (kept == total) ++nf;
                    else if (kept > 0) ++np;
                }
            }
            full[r * N + d] = nf;
            partial[r * N + d] = np;
        }
    }
}

/* Closed forms for T = Tq = Tk dividing L (n = L / T tiles per stripe):
 *  striped:    every (r, d) processes n(n-1)/2 full tiles below the
 *              diagonal and n diagonal tiles; a diagonal tile keeps j <= i
 *              when e <= d and j < i when e > d, so for T >= 2 it is
 *              partial, and for T = 1 it is full (e <= d) or empty (e > d).
 *  contiguous: e < d: n^2 full; e == d: n(n-1)/2 full + n diagonal tiles
 *              (partial for T >= 2, full for T = 1); e > d: nothing.
 *  zig-zag (T dividing C = S/(2N), c = C/T tiles per chunk): a query chunk
 *              keeps a whole key chunk of lower index and the causal
 *              triangle of its own.  e == d: chunks (d,d) and (2N-1-d,
 *              2N-1-d) are triangles of c(c-1)/2 full + c diagonal tiles,
 *              (2N-1-d, d) is c^2 full; e != d: exactly two chunk pairs
 *              are kept in full (e < d: (d,e), (2N-1-d,e); e > d:
 *              (2N-1-d,e), (2N-1-d,2N-1-e)), so 2c^2 full tiles.         */
void oracle_tile_counts_closed(int64_t S, int N, int64_t T, int layout, int64_t *full,
                               int64_t *partial) {
    int64_t L = S / N, n = L / T;
    for (int r = 0; r < N; ++r) {
        for (int d = 0; d < N; ++d) {
            int e = ((d - r) % N + N) % N;
            int64_t nf = 0, np = 0;
            int diag_kept_all = (T == 1);
            if (layout == 2) {
                int64_t c = (S / (2 * (int64_t)N)) / T;
                if (e == d) {
                    nf = c * (c - 1) + c * c;
                    if (diag_kept_all) nf += 2 * c;
                    else np = 2 * c;
                } else {
                    nf = 2 * c * c;
                }
            } else if (layout == 0) {
                nf = n * (n - 1) / 2;
                if (T >= 2) np = n;
                else if (e <= d) nf += n;
            } else {
                if (e < d) nf = n * n;
                else if (e == d) {
                    nf = n * (n - 1) / 2;
                    if (diag_kept_all) nf += n;
                    else np = n;
                }
            }
            full[r * N + d] = nf;
            partial[r * N + d] = np;
        }
    }
}

/* Modelled ring critical path: each round lasts as long as its busiest
 * device, so the sum over rounds of the largest per-device tile count
 * (§Summary: "each round runs at the pace of the slowest device"). */
int64_t oracle_critical_path(const int64_t *full, const int64_t *partial, int N) {
    int64_t total = 0;
    for (int r = 0; r < N; ++r) {
        int64_t mx = 0;
        for (int d = 0; d < N; ++d) {
            int64_t c = full[r * N + d] + partial[r * N + d];
            if (c > mx) mx = c;
        }
        total += mx;
    }
    return total;
}
