/*
 * gdn_oracle.c -- float64 CPU oracle for speculative-tree verification through a
 * Gated Delta Net layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file.  It shares no code, header, table or helper
 * with the CUDA library; the product path never calls it.
 *
 * What it computes (and where the pages state it):
 *   - Gated delta rule, "Trees from Marginals" (gist.science Technical Summary,
 *     section 3 "Rollback-Free Tree Verification for GDN", Challenge): the state
 *     update with alpha_t = exp(g_t).  This file keeps the state as S[d_v][d_k]
 *     so that one step reads
 *         S <- exp(g) * S * (I - beta k k^T) + beta v k^T,   o = scale * S q
 *     (the transpose of the page's d_k x d_v form; outputs are identical).
 *   - Tree semantics, same section, Solution bullets: the tree is sorted
 *     topologically (parent before child) and every node's output is the output
 *     of the recurrence run along its own root-to-node path, starting from the
 *     committed state S0, which is never modified.
 *   - Commit, same section, last bullet: once the accepted branch is known the
 *     state is advanced along that branch only.
 *
 * The oracle replays each node's whole path from S0, sequentially, in float64,
 * without sharing any prefix work between nodes.  It is deliberately slow.
 * Inputs arrive already upcast to double from their stored precision.
 *
 * Layouts (row-major, T = total nodes):
 *   q, k [T][Hk][d_k]; v [T][Hv][d_v]; g, beta [T][Hv]; S0 [B][Hv][d_v][d_k];
 *   parent [T] request-local (-1 = child of S0); offsets [B+1].
 *   Value head h reads key head h / (Hv / Hk).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t B, Hk, Hv, dk, dv;
    const int32_t *offsets, *parent;
    const double *q, *k, *v, *g, *beta, *S0;
    double scale;
} problem_t;

/* ------------------------------------------------------------------------ */
/* tree descriptor: ancestor bitmask (bit j of row i set iff j lies on i's    */
/* root-to-node path, i included) and depth (nodes on that path, root = 1).   */
/* Returns 0, or 1 if some parent[i] is outside [-1, i).                       */
/* ------------------------------------------------------------------------ */
int gdn_oracle_build_desc(const int32_t *parent, const int32_t *offsets, int32_t B,
                          int32_t words, uint32_t *mask, int32_t *depth)
{
    int bad = 0;
    for (int32_t b = 0; b < B; ++b) {
        int32_t lo = offsets[b], n = offsets[b + 1] - offsets[b];
        for (int32_t i = 0; i < n; ++i) {
            uint32_t *row = mask + (int64_t)(lo + i) * words;
            memset(row, 0, sizeof(uint32_t) * (size_t)words);
            int32_t d = 0, j = i, ok = 1;
            while (j >= 0) {                       /* walk parent pointers to the root */
                if (j >= words * 32) { ok = 0; break; }
                row[j >> 5] |= 1u << (j & 31);
                ++d;
                int32_t p = parent[lo + j];
                if (p < -1 || p >= j) { ok = 0; break; }
                j = p;
            }
            if (!ok) { bad = 1; memset(row, 0, sizeof(uint32_t) * (size_t)words); d = 0; }
            depth[lo + i] = d;
        }
    }
    return bad;
}

/* Root-to-node path of local node i (root first).  Returns its length, or -1. */
static int32_t path_of(const int32_t *parent_local, int32_t i, int32_t *path)
{
    int32_t len = 0, j = i;
    while (j >= 0) {
        path[len++] = j;
        int32_t p = parent_local[j];
        if (p < -1 || p >= j) return -1;
        j = p;
    }
    for (int32_t a = 0, b = len - 1; a < b; ++a, --b) {
        int32_t t = path[a]; path[a] = path[b]; path[b] = t;
    }
    return len;
}

/* One gated-delta-rule step on S[dv][dk] for token t of value head h. */
static void gdn_step(const problem_t *P, double *S, double *Sk, int64_t t, int32_t h)
{
    const int32_t hk = h / (P->Hv / P->Hk);
    const double *kt = P->k + (t * P->Hk + hk) * P->dk;
    const double *vt = P->v + (t * P->Hv + h) * P->dv;
    const double alpha = exp(P->g[t * P->Hv + h]);
    const double beta = P->beta[t * P->Hv + h];
    /* S (I - beta k k^T) = S - beta (S k) k^T */
    for (int32_t n = 0; n < P->dv; ++n) {
        double acc = 0.0;
        for (int32_t m = 0; m < P->dk; ++m) acc += S[n * P->dk + m] * kt[m];
        Sk[n] = acc;
    }
    for (int32_t n = 0; n < P->dv; ++n)
        for (int32_t m = 0; m < P->dk; ++m)
            S[n * P->dk + m] = alpha * (S[n * P->dk + m] - beta * Sk[n] * kt[m])
                               + beta * vt[n] * kt[m];
}

/* Walk node i of request b, value head h, from S0; leaves the state in S.
   Returns the path length or -1 on a malformed tree. */
static int32_t walk(const problem_t *P, int32_t b, int32_t h, int32_t i, double *S,
                    double *Sk, int32_t *path)
{
    const int32_t lo = P->offsets[b];
    const int64_t sz = (int64_t)P->dv * P->dk;
    memcpy(S, P->S0 + ((int64_t)b * P->Hv + h) * sz, sizeof(double) * (size_t)sz);
    int32_t len = path_of(P->parent + lo, i, path);
    for (int32_t s = 0; s < len; ++s) gdn_step(P, S, Sk, (int64_t)lo + path[s], h);
    return len;
}

static void readout(const problem_t *P, const double *S, int64_t t, int32_t h, double *out)
{
    const int32_t hk = h / (P->Hv / P->Hk);
    const double *qt = P->q + (t * P->Hk + hk) * P->dk;
    for (int32_t n = 0; n < P->dv; ++n) {
        double acc = 0.0;
        for (int32_t m = 0; m < P->dk; ++m) acc += S[n * P->dk + m] * qt[m];
        out[n] = P->scale * acc;
    }
}

/* ------------------------------------------------------------------------ */
/* work distribution over (request, value head) units                         */
/* ------------------------------------------------------------------------ */
typedef struct {
    const problem_t *P;
    int mode;                 /* 0 verify all, 1 selected nodes, 2 commit */
    double *out;
    const int64_t *sel; int64_t nsel;
    const int32_t *poff, *pidx;
    int64_t next;             /* shared counter, guarded by lock */
    int64_t nunits;
    int32_t status;
    pthread_mutex_t lock;
} job_t;

static int64_t take(job_t *J)
{
    pthread_mutex_lock(&J->lock);
    int64_t u = J->next < J->nunits ? J->next++ : -1;
    pthread_mutex_unlock(&J->lock);
    return u;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const problem_t *P = J->P;
    const int64_t sz = (int64_t)P->dv * P->dk;
    int32_t nmax = 1;
    for (int32_t b = 0; b < P->B; ++b) {
        int32_t n = P->offsets[b + 1] - P->offsets[b];
        if (n > nmax) nmax = n;
    }
    double *S = (double *)malloc(sizeof(double) * (size_t)sz);
    double *Sk = (double *)malloc(sizeof(double) * (size_t)P->dv);
    int32_t *path = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nmax + 1));
    int64_t u;
    while ((u = take(J)) >= 0) {
        if (J->mode == 0) {                      /* unit = (b, h) */
            int32_t b = (int32_t)(u / P->Hv), h = (int32_t)(u % P->Hv);
            int32_t lo = P->offsets[b], n = P->offsets[b + 1] - lo;
            for (int32_t i = 0; i < n; ++i) {
                if (walk(P, b, h, i, S, Sk, path) < 0) { J->status = 1; continue; }
                readout(P, S, (int64_t)lo + i, h, J->out + ((int64_t)(lo + i) * P->Hv + h) * P->dv);
            }
        } else if (J->mode == 1) {               /* unit = one selected (b, h, i) */
            int32_t b = (int32_t)J->sel[3 * u], h = (int32_t)J->sel[3 * u + 1];
            int32_t i = (int32_t)J->sel[3 * u + 2];
            if (walk(P, b, h, i, S, Sk, path) < 0) { J->status = 1; continue; }
            readout(P, S, (int64_t)P->offsets[b] + i, h, J->out + u * P->dv);
        } else {                                 /* unit = (b, h): commit the accepted path */
            int32_t b = (int32_t)(u / P->Hv), h = (int32_t)(u % P->Hv);
            int32_t lo = P->offsets[b];
            memcpy(S, P->S0 + ((int64_t)b * P->Hv + h) * sz, sizeof(double) * (size_t)sz);
            int32_t prev = -1;
            for (int32_t s = J->poff[b]; s < J->poff[b + 1]; ++s) {
                int32_t node = J->pidx[s];
                int32_t n = P->offsets[b + 1] - lo;
                if (node < 0 || node >= n || P->parent[lo + node] != prev) { J->status = 2; break; }
                gdn_step(P, S, Sk, (int64_t)lo + node, h);
                prev = node;
            }
            memcpy(J->out + ((int64_t)b * P->Hv + h) * sz, S, sizeof(double) * (size_t)sz);
        }
    }
    free(S); free(Sk); free(path);
    return NULL;
}

static int32_t run(job_t *J, int32_t nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    pthread_mutex_init(&J->lock, NULL);
    J->next = 0;
    J->status = 0;
    for (int32_t t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, J);
    worker(J);
    for (int32_t t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&J->lock);
    return J->status;
}

#define PROBLEM(P) problem_t P = { B, Hk, Hv, dk, dv, offsets, parent, q, k, v, g, beta, S0, scale }

/* o [T][Hv][dv]: every node's output.  Returns 0, or 1 on a malformed tree. */
int32_t gdn_oracle_verify(int32_t B, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                          const int32_t *offsets, const int32_t *parent, const double *q,
                          const double *k, const double *v, const double *g,
                          const double *beta, const double *S0, double scale, double *o,
                          int32_t nthreads)
{
    PROBLEM(P);
    job_t J; memset(&J, 0, sizeof J);
    J.P = &P; J.mode = 0; J.out = o; J.nunits = (int64_t)B * Hv;
    return run(&J, nthreads);
}

/* o_sel [nsel][dv]: outputs of the selected (b, h, i) triples only. */
int32_t gdn_oracle_verify_sel(int32_t B, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                              const int32_t *offsets, const int32_t *parent, const double *q,
                              const double *k, const double *v, const double *g,
                              const double *beta, const double *S0, double scale,
                              const int64_t *sel, int64_t nsel, double *o_sel, int32_t nthreads)
{
    PROBLEM(P);
    job_t J; memset(&J, 0, sizeof J);
    J.P = &P; J.mode = 1; J.out = o_sel; J.sel = sel; J.nsel = nsel; J.nunits = nsel;
    return run(&J, nthreads);
}

/* S_new [B][Hv][dv][dk]: the state after the accepted path of each request
   (root first; an empty path leaves S0).  Returns 0, or 2 on a path that does
   not start at a root or does not follow parent -> child edges. */
int32_t gdn_oracle_commit(int32_t B, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                          const int32_t *offsets, const int32_t *parent, const double *k,
                          const double *v, const double *g, const double *beta,
                          const double *S0, const int32_t *path_offsets,
                          const int32_t *path_idx, double *S_new, int32_t nthreads)
{
    const double *q = NULL;
    double scale = 1.0;
    PROBLEM(P);
    job_t J; memset(&J, 0, sizeof J);
    J.P = &P; J.mode = 2; J.out = S_new; J.poff = path_offsets; J.pidx = path_idx;
    J.nunits = (int64_t)B * Hv;
    return run(&J, nthreads);
}

/* The walked state at node i of request b, value head h (S [dv][dk]). */
int32_t gdn_oracle_state_at(int32_t B, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                            const int32_t *offsets, const int32_t *parent, const double *k,
                            const double *v, const double *g, const double *beta,
                            const double *S0, int32_t b, int32_t h, int32_t i, double *S)
{
    const double *q = NULL;
    double scale = 1.0;
    PROBLEM(P);
    double *Sk = (double *)malloc(sizeof(double) * (size_t)dv);
    int32_t n = offsets[b + 1] - offsets[b];
    int32_t *path = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int32_t r = walk(&P, b, h, i, S, Sk, path);
    free(Sk); free(path);
    return r < 0 ? 1 : 0;
}
