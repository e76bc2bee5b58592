/*
 * CPU oracle for closed-form Gated DeltaNet tree verification -- TEST
 * INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file; the product path never does.  It shares no
 * code, header or constant with the CUDA path.
 *
 * It computes, in double precision and node by node, what the closed form of
 * "Bole: Efficient Tree Speculation for Hybrid-Attention Language Models"
 * (Theorem 1) is proven to equal: sequential execution of the gated delta
 * rule along every root-to-node path, with a full state snapshot per node.
 *
 *   GDN recurrence (Section II-A, Eq. (1)), for node t with parent pi(t):
 *     S~_t = gamma_t * S_pi(t)          (S_pi(t) = S_pre at the committed root)
 *     u_t  = beta_t * (v_t - S~_t^T k_t)
 *     S_t  = S~_t + k_t u_t^T
 *     o_t  = S_t^T q_t                   (read-out of the post-update state)
 *   Cumulative decay (Lemma 1, Eq. (4)): P_t = prod of gamma over the
 *     ancestors-or-self of t; reported as log P_t.
 *   Ancestor mask (Section II-B / Lemma 2): a node sees the committed prefix
 *     and its own proposal ancestors only, never a sibling branch.
 *   Commit (factorized speculative state, Eq. (10)): the committed state after
 *     acceptance equals the state reached by the accepted node a, i.e. S_a;
 *     with no accepted node the slot keeps S_pre.
 *
 * Layouts match the library's: offsets [B+1], parent [N] (request-local,
 * -1 = committed root), q/k [N,H,dk], v [N,H,dv], gamma/beta [N,H],
 * S_pre/S_new [B,H,dk,dv] (dv contiguous), O/U [N,H,dv], logP [N,H].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_TOPOLOGY 3
#define ORACLE_DEPTH 4
#define ORACLE_NOMEM 9
#define ORACLE_MAX_TREE 128

/* ------------------------------------------------------------------------ */
/* topology: depth, ancestor-or-self bit masks, per-request maximum depth    */
/* ------------------------------------------------------------------------ */

int oracle_pack(int B, const int32_t *offsets, const int32_t *parent, int max_depth,
                int32_t *depth, uint32_t *anc, int32_t *req_depth)
{
    for (int b = 0; b < B; ++b) {
        int o = offsets[b], T = offsets[b + 1] - offsets[b];
        if (T < 0 || T > ORACLE_MAX_TREE) return ORACLE_BAD_TOPOLOGY;
        int dmax = 0;
        for (int i = 0; i < T; ++i) {
            int p = parent[o + i];
            if (p < -1 || p >= i) return ORACLE_BAD_TOPOLOGY;
            /* walk up the parent links: every visited node is an ancestor */
            uint32_t m[4] = {0, 0, 0, 0};
            int d = -1;
            for (int j = i; j != -1; j = parent[o + j]) {
                m[j >> 5] |= 1u << (j & 31);
                ++d;
            }
            for (int w = 0; w < 4; ++w) anc[(size_t)(o + i) * 4 + w] = m[w];
            depth[o + i] = d;
            if (d > dmax) dmax = d;
        }
        req_depth[b] = dmax;
        if (dmax > max_depth) return ORACLE_DEPTH;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* verification: per (request, head) unit, sequential tree execution         */
/* ------------------------------------------------------------------------ */

typedef struct {
    int B, H, dk, dv;
    const int32_t *offsets, *parent, *accepted;
    const double *S_pre, *q, *k, *v, *gamma, *beta;
    double *O, *U, *logP, *S_new;
    int unit_begin, unit_end;
    int next; /* shared work counter */
    int status;
} job_t;

/* One unit of the verification: tree b, head h. */
static int verify_unit(job_t *J, int b, int h, double *snap, double *P)
{
    const int H = J->H, dk = J->dk, dv = J->dv;
    const int o = J->offsets[b], T = J->offsets[b + 1] - o;
    const double *S0 = J->S_pre + ((size_t)b * H + h) * dk * dv;
    for (int i = 0; i < T; ++i) {
        const size_t nh = (size_t)(o + i) * H + h;
        const int p = J->parent[o + i];
        const double *Sp = (p < 0) ? S0 : snap + (size_t)p * dk * dv;
        double *Si = snap + (size_t)i * dk * dv;
        const double g = J->gamma[nh], bt = J->beta[nh];
        const double *q = J->q + nh * dk, *k = J->k + nh * dk, *v = J->v + nh * dv;
        double *u = J->U + nh * dv, *out = J->O + nh * dv;
        /* S~ = gamma * S_parent */
        for (size_t e = 0; e < (size_t)dk * dv; ++e) Si[e] = g * Sp[e];
        /* u = beta * (v - S~^T k) */
        for (int c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int r = 0; r < dk; ++r) acc += Si[(size_t)r * dv + c] * k[r];
            u[c] = bt * (v[c] - acc);
        }
        /* S = S~ + k u^T */
        for (int r = 0; r < dk; ++r)
            for (int c = 0; c < dv; ++c) Si[(size_t)r * dv + c] += k[r] * u[c];
        /* o = S^T q */
        for (int c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int r = 0; r < dk; ++r) acc += Si[(size_t)r * dv + c] * q[r];
            out[c] = acc;
        }
        /* cumulative decay along the parent link */
        P[i] = g * (p < 0 ? 1.0 : P[p]);
        J->logP[nh] = log(P[i]);
    }
    return ORACLE_OK;
}

/* Commit for tree b, head h: replay the accepted root-to-a path only. */
static int commit_unit(job_t *J, int b, int h, double *S, double *tmp)
{
    const int H = J->H, dk = J->dk, dv = J->dv;
    const int o = J->offsets[b], T = J->offsets[b + 1] - o;
    const double *S0 = J->S_pre + ((size_t)b * H + h) * dk * dv;
    double *Sout = J->S_new + ((size_t)b * H + h) * dk * dv;
    memcpy(S, S0, sizeof(double) * dk * dv);
    const int a = J->accepted[b];
    if (a >= 0 && a < T) {
        int path[ORACLE_MAX_TREE];
        int L = 0;
        for (int j = a; j != -1; j = J->parent[o + j]) path[L++] = j;
        for (int t = L - 1; t >= 0; --t) {
            const size_t nh = (size_t)(o + path[t]) * H + h;
            const double g = J->gamma[nh], bt = J->beta[nh];
            const double *k = J->k + nh * dk, *v = J->v + nh * dv;
            for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] *= g;
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int r = 0; r < dk; ++r) acc += S[(size_t)r * dv + c] * k[r];
                tmp[c] = bt * (v[c] - acc);
            }
            for (int r = 0; r < dk; ++r)
                for (int c = 0; c < dv; ++c) S[(size_t)r * dv + c] += k[r] * tmp[c];
        }
    }
    memcpy(Sout, S, sizeof(double) * dk * dv);
    return ORACLE_OK;
}

static void *verify_worker(void *arg)
{
    job_t *J = (job_t *)arg;
    int Tmax = 0;
    for (int b = 0; b < J->B; ++b) {
        int T = J->offsets[b + 1] - J->offsets[b];
        if (T > Tmax) Tmax = T;
    }
    double *snap = (double *)malloc(sizeof(double) * (size_t)(Tmax > 0 ? Tmax : 1) * J->dk * J->dv);
    double *P = (double *)malloc(sizeof(double) * (size_t)(Tmax > 0 ? Tmax : 1));
    if (!snap || !P) {
        free(snap); free(P);
        __atomic_store_n(&J->status, ORACLE_NOMEM, __ATOMIC_RELAXED);
        return NULL;
    }
    for (;;) {
        int w = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED) + J->unit_begin;
        if (w >= J->unit_end) break;
        verify_unit(J, w / J->H, w % J->H, snap, P);
    }
    free(snap); free(P);
    return NULL;
}

static void *commit_worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->dk * J->dv);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!S || !tmp) {
        free(S); free(tmp);
        __atomic_store_n(&J->status, ORACLE_NOMEM, __ATOMIC_RELAXED);
        return NULL;
    }
    for (;;) {
        int w = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED) + J->unit_begin;
        if (w >= J->unit_end) break;
        commit_unit(J, w / J->H, w % J->H, S, tmp);
    }
    free(S); free(tmp);
    return NULL;
}

static int run_threads(job_t *J, void *(*fn)(void *), int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, fn, J) != 0) break;
        ++started;
    }
    fn(J);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    return J->status;
}

static int check_topology(int B, const int32_t *offsets, const int32_t *parent)
{
    for (int b = 0; b < B; ++b) {
        int T = offsets[b + 1] - offsets[b];
        if (T < 0 || T > ORACLE_MAX_TREE) return ORACLE_BAD_TOPOLOGY;
        for (int i = 0; i < T; ++i) {
            int p = parent[offsets[b] + i];
            if (p < -1 || p >= i) return ORACLE_BAD_TOPOLOGY;
        }
    }
    return ORACLE_OK;
}

/* Units are numbered w = b * H + h; [unit_begin, unit_end) selects a slice.
 * Outputs of units outside the slice are left untouched. */
int oracle_verify(int B, int H, int dk, int dv, const int32_t *offsets, const int32_t *parent,
                  const double *S_pre, const double *q, const double *k, const double *v,
                  const double *gamma, const double *beta, double *O, double *U, double *logP,
                  int unit_begin, int unit_end, int nthreads)
{
    int s = check_topology(B, offsets, parent);
    if (s != ORACLE_OK) return s;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.H = H; J.dk = dk; J.dv = dv;
    J.offsets = offsets; J.parent = parent;
    J.S_pre = S_pre; J.q = q; J.k = k; J.v = v; J.gamma = gamma; J.beta = beta;
    J.O = O; J.U = U; J.logP = logP;
    J.unit_begin = unit_begin < 0 ? 0 : unit_begin;
    J.unit_end = (unit_end < 0 || unit_end > B * H) ? B * H : unit_end;
    return run_threads(&J, verify_worker, nthreads);
}

int oracle_commit(int B, int H, int dk, int dv, const int32_t *offsets, const int32_t *parent,
                  const int32_t *accepted, const double *S_pre, const double *k, const double *v,
                  const double *gamma, const double *beta, double *S_new, int unit_begin,
                  int unit_end, int nthreads)
{
    int s = check_topology(B, offsets, parent);
    if (s != ORACLE_OK) return s;
    for (int b = 0; b < B; ++b) {
        int T = offsets[b + 1] - offsets[b];
        if (accepted[b] < -1 || accepted[b] >= T) return ORACLE_BAD_TOPOLOGY;
    }
    job_t J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.H = H; J.dk = dk; J.dv = dv;
    J.offsets = offsets; J.parent = parent; J.accepted = accepted;
    J.S_pre = S_pre; J.k = k; J.v = v; J.gamma = gamma; J.beta = beta;
    J.S_new = S_new;
    J.unit_begin = unit_begin < 0 ? 0 : unit_begin;
    J.unit_end = (unit_end < 0 || unit_end > B * H) ? B * H : unit_end;
    return run_threads(&J, commit_worker, nthreads);
}
