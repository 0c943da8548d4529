/*
 * FP64 CPU oracle for the gated delta rule (DeltaNet / Gated DeltaNet / KDA).
 *
 * TEST INFRASTRUCTURE ONLY. This file is used by the test-suite, by the smoke
 * check and by the benchmark's CPU-baseline leg. The product path never loads
 * it, and it shares no code with the CUDA library.
 *
 * What it computes: the token-by-token recurrence of "Kimi Delta Attention"
 * (mainlymatmul.com/blog/kimi-delta-attention, section 4, boxed KDA update;
 * the same five steps in the [K,V] state layout are printed at the end of that
 * section), for one head and one sequence at a time, state S in R^{K x V}:
 *
 *     a_t  = exp(g_t)                  (per key channel; scalar g broadcast;
 *                                       a_t = 1 when there is no gate)
 *     S~   = diag(a_t) S_{t-1}         forget each key channel (before predict)
 *     p_t  = S~^T k_t                  predict
 *     r_t  = beta_t (v_t - p_t)        correct
 *     S_t  = S~ + k_t r_t^T            write
 *     o_t  = S_t^T (scale q_t)         read, after the write
 *
 * GatedDeltaNet-2 ("GatedDeltaNet-2 (NVlabs) — official spec transcription",
 * §3, the per-token body) replaces the scalar beta by an erase vector b on the
 * key axis and a write vector w on the value axis:
 *
 *     p_t  = S~^T (b_t .* k_t)         erase
 *     r_t  = w_t .* v_t - p_t          write value
 *
 * (b = w = beta 1 gives the rule above), with the same write and read steps.
 *
 * with S_{-1} = h0 (or 0) and ht = S_{L-1}. The operator family is the gate
 * choice of the ReWY paper's Table 1 (hub.valency.io W_esyzsyuq, "Delta-rule
 * operators"): DeltaNet has no decay, GDN a scalar decay, KDA a vector decay.
 *
 * The backward pass is back-propagation through time of exactly those steps,
 * derived by hand (reverse mode, one step at a time, in reverse order):
 *
 *     read:     dq_t   = scale * S_t do_t ;        Sbar += scale q_t do_t^T
 *     write:    dk_t   = Sbar r_t ;                rbar  = Sbar^T k_t
 *     correct:  dv_t   = beta_t rbar ;             dbeta_t = <rbar, v_t - p_t>
 *               pbar   = -beta_t rbar
 *     predict:  S~bar  = Sbar + k_t pbar^T ;       dk_t += S~ pbar
 *     forget:   dg_t   = rowsum(S~bar .* S~)  (d a / d g = a is folded in;
 *                                              scalar gate: summed over K)
 *               Sbar   = diag(a_t) S~bar
 *
 * and for GatedDeltaNet-2, in place of the correct and predict lines:
 *
 *     correct:  dv_t = w_t .* rbar ;   dw_t = rbar .* v_t ;   pbar = -rbar
 *     predict:  S~bar = Sbar + (b_t .* k_t) pbar^T ;  u = S~ pbar ;
 *               db_t = k_t .* u ;      dk_t += b_t .* u
 *
 * starting from Sbar = dht (or 0); after the first token dh0 = Sbar. The loss
 * whose gradients these are is <do, o> + <dht, ht>.
 *
 * Memory: the forward keeps one copy of S every 64 tokens; the reverse pass
 * recomputes each 64-token segment from its copy. Work items are
 * (sequence, head) pairs, split statically over threads, so the result does
 * not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SEG 64

typedef struct {
    int n_seq;               /* number of sequences */
    const int64_t *seq_start;/* n_seq + 1 token offsets into the packed token axis */
    int H, K, V;
    int gate;                /* 0 none, 1 scalar [T,H], 2 per channel [T,H,K] */
    double scale;
    const double *q, *k;     /* [T, H, K] */
    const double *v;         /* [T, H, V] */
    const double *beta;      /* [T, H] */
    const double *g;         /* see gate; NULL when gate == 0 */
    const double *h0;        /* [n_seq, H, K, V] or NULL (zeros) */
    const double *dout;      /* [T, H, V] (backward only) */
    const double *dht;       /* [n_seq, H, K, V] or NULL (zeros) */
    double *o;               /* [T, H, V] */
    double *ht;              /* [n_seq, H, K, V] or NULL */
    double *dq, *dk, *dv, *dbeta, *dg, *dh0; /* backward outputs; dg NULL iff gate == 0 */
    int backward;
    const int32_t *items;    /* optional list of (seq, head) pairs, 2 ints each */
    int n_items;             /* number of pairs in items (0: all pairs) */
    const double *erase;     /* [T, H, K] or NULL: GatedDeltaNet-2 erase vector (beta unused) */
    const double *write;     /* [T, H, V]: GatedDeltaNet-2 write vector (with erase) */
    double *derase, *dwrite; /* their gradients (backward, with erase) */
} oracle_problem;

typedef struct {
    const oracle_problem *p;
    int tid, nthreads;
    int status;
} worker_arg;

/* decay factors a_t for token t (global index) and head h into a[K] */
static void decay(const oracle_problem *p, int64_t t, int h, double *a) {
    int K = p->K;
    if (p->gate == 0) {
        for (int i = 0; i < K; ++i) a[i] = 1.0;
    } else if (p->gate == 1) {
        double e = exp(p->g[t * p->H + h]);
        for (int i = 0; i < K; ++i) a[i] = e;
    } else {
        const double *gt = p->g + (t * p->H + h) * (int64_t)K;
        for (int i = 0; i < K; ++i) a[i] = exp(gt[i]);
    }
}

/* One forward step: S (in: S_{t-1}, out: S_t). Writes o_t when o != NULL. */
static void step_fwd(const oracle_problem *p, int64_t t, int h, double *S, double *a,
                     double *pv, double *r, double *o) {
    int K = p->K, V = p->V, H = p->H;
    const double *kt = p->k + (t * H + h) * (int64_t)K;
    const double *qt = p->q + (t * H + h) * (int64_t)K;
    const double *vt = p->v + (t * H + h) * (int64_t)V;
    const double *bv = p->erase ? p->erase + (t * H + h) * (int64_t)K : NULL;
    const double *wv = p->erase ? p->write + (t * H + h) * (int64_t)V : NULL;
    double bt = p->erase ? 0.0 : p->beta[t * H + h];
    decay(p, t, h, a);
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) S[i * V + j] *= a[i];
    for (int j = 0; j < V; ++j) pv[j] = 0.0;
    for (int i = 0; i < K; ++i) {
        double ke = bv ? bv[i] * kt[i] : kt[i];
        for (int j = 0; j < V; ++j) pv[j] += S[i * V + j] * ke;
    }
    for (int j = 0; j < V; ++j) r[j] = bv ? wv[j] * vt[j] - pv[j] : bt * (vt[j] - pv[j]);
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) S[i * V + j] += kt[i] * r[j];
    if (o) {
        for (int j = 0; j < V; ++j) o[j] = 0.0;
        for (int i = 0; i < K; ++i) {
            double sq = p->scale * qt[i];
            for (int j = 0; j < V; ++j) o[j] += S[i * V + j] * sq;
        }
    }
}

/* Reverse step for token t. Sprev = S_{t-1}. Sbar holds the adjoint of S_t on
 * entry and the adjoint of S_{t-1} on exit. */
static void step_bwd(const oracle_problem *p, int64_t t, int h, const double *Sprev,
                     double *Sbar, double *St, double *a, double *pv, double *r,
                     double *rbar) {
    int K = p->K, V = p->V, H = p->H;
    const double *kt = p->k + (t * H + h) * (int64_t)K;
    const double *qt = p->q + (t * H + h) * (int64_t)K;
    const double *vt = p->v + (t * H + h) * (int64_t)V;
    const double *dot = p->dout + (t * H + h) * (int64_t)V;
    const double *bv = p->erase ? p->erase + (t * H + h) * (int64_t)K : NULL;
    const double *wv = p->erase ? p->write + (t * H + h) * (int64_t)V : NULL;
    double bt = p->erase ? 0.0 : p->beta[t * H + h];
    double *dqt = p->dq + (t * H + h) * (int64_t)K;
    double *dkt = p->dk + (t * H + h) * (int64_t)K;
    double *dvt = p->dv + (t * H + h) * (int64_t)V;

    /* recompute the forward quantities of this step */
    decay(p, t, h, a);
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) St[i * V + j] = a[i] * Sprev[i * V + j];   /* S~ */
    for (int j = 0; j < V; ++j) pv[j] = 0.0;
    for (int i = 0; i < K; ++i) {
        double ke = bv ? bv[i] * kt[i] : kt[i];
        for (int j = 0; j < V; ++j) pv[j] += St[i * V + j] * ke;
    }
    for (int j = 0; j < V; ++j) r[j] = bv ? wv[j] * vt[j] - pv[j] : bt * (vt[j] - pv[j]);

    /* read: o = S_t^T (scale q), S_t = S~ + k r^T */
    for (int i = 0; i < K; ++i) {
        double acc = 0.0;
        for (int j = 0; j < V; ++j) acc += (St[i * V + j] + kt[i] * r[j]) * dot[j];
        dqt[i] = p->scale * acc;
    }
    for (int i = 0; i < K; ++i) {
        double sq = p->scale * qt[i];
        for (int j = 0; j < V; ++j) Sbar[i * V + j] += sq * dot[j];
    }
    /* write: S_t = S~ + k r^T */
    for (int i = 0; i < K; ++i) {
        double acc = 0.0;
        for (int j = 0; j < V; ++j) acc += Sbar[i * V + j] * r[j];
        dkt[i] = acc;
    }
    for (int j = 0; j < V; ++j) rbar[j] = 0.0;
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) rbar[j] += Sbar[i * V + j] * kt[i];
    if (bv) {
        /* correct: r = w .* v - p */
        double *dwt = p->dwrite + (t * H + h) * (int64_t)V;
        double *dbt = p->derase + (t * H + h) * (int64_t)K;
        for (int j = 0; j < V; ++j) {
            dvt[j] = wv[j] * rbar[j];
            dwt[j] = rbar[j] * vt[j];
            rbar[j] = -rbar[j];                          /* pbar */
        }
        /* erase: p = S~^T (b .* k) */
        for (int i = 0; i < K; ++i) {
            double u = 0.0, ke = bv[i] * kt[i];
            for (int j = 0; j < V; ++j) {
                Sbar[i * V + j] += ke * rbar[j];         /* S~bar */
                u += St[i * V + j] * rbar[j];
            }
            dbt[i] = kt[i] * u;
            dkt[i] += bv[i] * u;
        }
    } else {
        /* correct: r = beta (v - p) */
        double db = 0.0;
        for (int j = 0; j < V; ++j) {
            dvt[j] = bt * rbar[j];
            db += rbar[j] * (vt[j] - pv[j]);
        }
        p->dbeta[t * H + h] = db;
        /* predict: p = S~^T k ; pbar = -beta rbar (reuse rbar as pbar) */
        for (int j = 0; j < V; ++j) rbar[j] = -bt * rbar[j];
        for (int i = 0; i < K; ++i) {
            double acc = 0.0;
            for (int j = 0; j < V; ++j) {
                Sbar[i * V + j] += kt[i] * rbar[j];      /* S~bar */
                acc += St[i * V + j] * rbar[j];
            }
            dkt[i] += acc;
        }
    }
    /* forget: S~ = diag(a) S_{t-1} */
    if (p->gate == 2) {
        double *dgt = p->dg + (t * H + h) * (int64_t)K;
        for (int i = 0; i < K; ++i) {
            double acc = 0.0;
            for (int j = 0; j < V; ++j) acc += Sbar[i * V + j] * St[i * V + j];
            dgt[i] = acc;
        }
    } else if (p->gate == 1) {
        double acc = 0.0;
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < V; ++j) acc += Sbar[i * V + j] * St[i * V + j];
        p->dg[t * H + h] = acc;
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) Sbar[i * V + j] *= a[i];
}

static int run_pair(const oracle_problem *p, int n, int h) {
    int K = p->K, V = p->V, H = p->H;
    int64_t t0 = p->seq_start[n], t1 = p->seq_start[n + 1];
    int64_t L = t1 - t0;
    int64_t KV = (int64_t)K * V;
    int64_t nseg = (L + SEG - 1) / SEG;
    double *S = (double *)malloc(sizeof(double) * KV);
    double *ck = (double *)malloc(sizeof(double) * KV * (nseg > 0 ? nseg : 1));
    double *a = (double *)malloc(sizeof(double) * K);
    double *pv = (double *)malloc(sizeof(double) * V);
    double *r = (double *)malloc(sizeof(double) * V);
    double *rb = (double *)malloc(sizeof(double) * V);
    if (!S || !ck || !a || !pv || !r || !rb) {
        free(S); free(ck); free(a); free(pv); free(r); free(rb);
        return 1;
    }
    const int64_t st_off = ((int64_t)n * H + h) * KV;
    if (p->h0) memcpy(S, p->h0 + st_off, sizeof(double) * KV);
    else memset(S, 0, sizeof(double) * KV);

    for (int64_t t = 0; t < L; ++t) {
        if (t % SEG == 0) memcpy(ck + (t / SEG) * KV, S, sizeof(double) * KV);
        step_fwd(p, t0 + t, h, S, a, pv, r, p->o + ((t0 + t) * H + h) * (int64_t)V);
    }
    if (p->ht) memcpy(p->ht + st_off, S, sizeof(double) * KV);

    int status = 0;
    if (p->backward) {
        double *Sbar = (double *)malloc(sizeof(double) * KV);
        double *St = (double *)malloc(sizeof(double) * KV);
        double *hist = (double *)malloc(sizeof(double) * KV * SEG);  /* S_{t-1} per token */
        if (!Sbar || !St || !hist) {
            status = 1;
        } else {
            if (p->dht) memcpy(Sbar, p->dht + st_off, sizeof(double) * KV);
            else memset(Sbar, 0, sizeof(double) * KV);
            for (int64_t s = nseg - 1; s >= 0; --s) {
                int64_t a0 = s * SEG, a1 = (a0 + SEG < L) ? a0 + SEG : L;
                memcpy(S, ck + s * KV, sizeof(double) * KV);
                for (int64_t t = a0; t < a1; ++t) {
                    memcpy(hist + (t - a0) * KV, S, sizeof(double) * KV);
                    step_fwd(p, t0 + t, h, S, a, pv, r, NULL);
                }
                for (int64_t t = a1 - 1; t >= a0; --t)
                    step_bwd(p, t0 + t, h, hist + (t - a0) * KV, Sbar, St, a, pv, r, rb);
            }
            if (p->dh0) memcpy(p->dh0 + st_off, Sbar, sizeof(double) * KV);
        }
        free(Sbar); free(St); free(hist);
    }
    free(S); free(ck); free(a); free(pv); free(r); free(rb);
    return status;
}

static void *worker(void *arg) {
    worker_arg *w = (worker_arg *)arg;
    const oracle_problem *p = w->p;
    int total = p->n_items > 0 ? p->n_items : p->n_seq * p->H;
    for (int i = w->tid; i < total; i += w->nthreads) {
        int n, h;
        if (p->n_items > 0) { n = p->items[2 * i]; h = p->items[2 * i + 1]; }
        else { n = i / p->H; h = i % p->H; }
        if (run_pair(p, n, h)) w->status = 1;
    }
    return NULL;
}

/* Runs the recurrence (and its reverse pass when p->backward) for every
 * (sequence, head) pair, or for the listed ones. Returns 0 on success, 1 on
 * an allocation failure, 2 on invalid arguments. */
int kda_oracle_run(const oracle_problem *p, int nthreads) {
    if (!p || p->n_seq < 0 || p->H <= 0 || p->K <= 0 || p->V <= 0 || !p->seq_start ||
        !p->q || !p->k || !p->v || (!p->beta && !p->erase) || (p->erase && !p->write) || !p->o ||
        (p->gate != 0 && !p->g) || p->gate < 0 || p->gate > 2)
        return 2;
    if (p->backward && (!p->dout || !p->dq || !p->dk || !p->dv || (!p->erase && !p->dbeta) ||
                        (p->erase && (!p->derase || !p->dwrite)) || (p->gate != 0 && !p->dg)))
        return 2;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    worker_arg wa[256];
    for (int i = 0; i < nthreads; ++i) {
        wa[i].p = p; wa[i].tid = i; wa[i].nthreads = nthreads; wa[i].status = 0;
    }
    if (nthreads == 1) {
        worker(&wa[0]);
        return wa[0].status;
    }
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &wa[i]) != 0) break;
        ++started;
    }
    /* threads that failed to start: run their share here */
    for (int i = started; i < nthreads; ++i) worker(&wa[i]);
    int status = 0;
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    for (int i = 0; i < nthreads; ++i) status |= wa[i].status;
    return status;
}

int kda_oracle_abi_version(void) { return 1; }
