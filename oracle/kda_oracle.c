/*
 * kda_oracle.c -- plain fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the CPU-baseline leg of
 * the benchmark are its only callers. The CUDA library never links, loads or calls this
 * file, and it shares no source, header, table or helper with the CUDA path.
 *
 * What the method computes, from the pages:
 *  - "Inside Kimi K3's Architecture" (maidul-haque blog), section "Kimi Delta Attention:
 *    the linear core": KDA keeps a fixed-size recurrent state; the delta rule removes the
 *    value that a key currently reads out of the state before the fresh value is written,
 *    and the forget gate decays the state per channel rather than with one scalar.
 *  - "Kimi K3 Explained" (researchpapers.dev), "Architecture at a glance" and the FAQ
 *    entry "What is Kimi Delta Attention?": a delta-rule recurrence with a channel-wise
 *    forget gate whose log-decay is bounded below through a scaled sigmoid.
 *
 * The plain reading of those sentences, per (sequence, head), with state S (d_k x d_v):
 *      S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *      o_t = S_t^T q_t,        alpha_t = exp(g_t)  (g_t: natural-log decay per key channel)
 * Order within a token: decay, then the delta correction against the decayed state, then the
 * write, then the read-out from the updated state. There is no scale on q.
 *
 * Functions (all fp64, all return 0 on success and a negative code on bad arguments):
 *  kda_oracle_recurrent  -- the recurrence above, token by token; the decode step is one
 *                           token of it. It applies (I - b k k^T) M as M - b k (k^T M),
 *                           which is the same product expanded (no other rewriting).
 *  kda_oracle_literal    -- the same recurrence with the d_k x d_k transition matrix
 *                           formed explicitly; O(d_k^2 d_v) per token, for small cases.
 *  kda_oracle_scaled_sigmoid_gate -- the log-decay from gate logits, g = -bound * sigmoid(x)
 *                           per element ("Kimi K3 Explained", researchpapers.dev, "Architecture
 *                           at a glance": the log-decay is bounded below through a scaled
 *                           sigmoid); the bound's value is not on the pages (the workloads use 5).
 *  kda_oracle_l2_normalize -- each row of d values divided by sqrt(sum of its squares + eps).
 *                           The pages do not describe this step; the workloads feed q and k as
 *                           unit vectors per (token, head), and the library can form them in its
 *                           kernels. The eps (1e-6 there) only keeps a zero row finite.
 *  kda_oracle_backward  -- gradients of L = sum(do * o) + sum(d_final * S_final) with respect
 *                           to q, k, v, g, beta and the initial state, by reverse-mode
 *                           differentiation of the recurrence token by token (the pages train
 *                           the model but give no gradient method; this is the adjoint of the
 *                           steps above, in reverse order: read-out, write, delta correction,
 *                           decay). The states before each token are kept from a forward pass.
 *  kda_oracle_output_gate -- y = o * sigmoid(z) per element: the output gate, an input-dependent
 *                           full-rank projection z ("Kimi K3 Explained", researchpapers.dev,
 *                           "Architecture at a glance"); the pages name no activation, the
 *                           logistic function is the plain reading.
 *  kda_oracle_chunked    -- a separately written chunkwise form of the same recurrence
 *                           (per-chunk cumulative log-decay, the strictly lower intra-chunk
 *                           matrix, a triangular solve for the delta corrections, one state
 *                           update per chunk). It is a check of the recurrence and a source
 *                           of per-stage intermediates; it is exact up to rounding and needs
 *                           chunk * max|g| < 700 so that exp(-cumsum g) stays finite in fp64.
 *
 * Layouts (row-major, contiguous): q, k, g [T_total, H, d_k]; v, o [T_total, H, d_v];
 * beta [T_total, H]; states [N, H, d_k, d_v]. Sequence n covers rows cu[n] .. cu[n+1]-1.
 * init_state may be NULL (zero state); final_state may be NULL.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_EBADARG (-1)
#define KDA_ORACLE_ENOMEM (-2)

typedef struct {
    int n_seqs, H, dk, dv;
    const int64_t *cu;
    const double *q, *k, *v, *g, *beta, *init;
    double *o, *fin;
} problem_t;

static int check_problem(const problem_t *p)
{
    if (p->n_seqs < 0 || p->H <= 0 || p->dk <= 0 || p->dv <= 0 || !p->cu) return KDA_ORACLE_EBADARG;
    for (int n = 0; n < p->n_seqs; ++n)
        if (p->cu[n + 1] < p->cu[n]) return KDA_ORACLE_EBADARG;
    if (p->cu[p->n_seqs] > p->cu[0] && (!p->q || !p->k || !p->v || !p->g || !p->beta || !p->o))
        return KDA_ORACLE_EBADARG;
    return 0;
}

/* Start state of (n, h): the caller's initial state or zeros. */
static void load_state(const problem_t *p, int n, int h, double *S)
{
    size_t sz = (size_t)p->dk * p->dv;
    if (p->init) memcpy(S, p->init + ((size_t)n * p->H + h) * sz, sz * sizeof(double));
    else memset(S, 0, sz * sizeof(double));
}

static void store_state(const problem_t *p, int n, int h, const double *S)
{
    size_t sz = (size_t)p->dk * p->dv;
    if (p->fin) memcpy(p->fin + ((size_t)n * p->H + h) * sz, S, sz * sizeof(double));
}

/* ---------------------------------------------------------------- recurrence ---------- */

/* One token of the recurrence on state S (dk x dv). u is dv scratch. */
static void recurrent_token(int dk, int dv, const double *q, const double *k, const double *v,
                            const double *g, double beta, double *S, double *o, double *u)
{
    /* Diag(alpha_t) S_{t-1}: row i of S is key channel i. */
    for (int i = 0; i < dk; ++i) {
        double a = exp(g[i]);
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;
    }
    /* (I - b k k^T) M + b k v^T = M + k (b (v - M^T k))^T with M the decayed state. */
    for (int j = 0; j < dv; ++j) {
        double kv = 0.0;
        for (int i = 0; i < dk; ++i) kv += S[(size_t)i * dv + j] * k[i];
        u[j] = beta * (v[j] - kv);
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += k[i] * u[j];
    /* o_t = S_t^T q_t */
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * q[i];
        o[j] = acc;
    }
}

static int run_recurrent(const problem_t *p, int n_threads)
{
    int err = check_problem(p);
    if (err) return err;
    const int H = p->H, dk = p->dk, dv = p->dv;
    const int pairs = p->n_seqs * H;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int ph = 0; ph < pairs; ++ph) {
        int n = ph / H, h = ph % H;
        double *S = malloc(sizeof(double) * ((size_t)dk * dv + dv));
        if (!S) { failed |= 1; continue; }
        double *u = S + (size_t)dk * dv;
        load_state(p, n, h, S);
        for (int64_t t = p->cu[n]; t < p->cu[n + 1]; ++t) {
            size_t r = (size_t)t * H + h;
            recurrent_token(dk, dv, p->q + r * dk, p->k + r * dk, p->v + r * dv, p->g + r * dk,
                            p->beta[r], S, p->o + r * dv, u);
        }
        store_state(p, n, h, S);
        free(S);
    }
    return failed ? KDA_ORACLE_ENOMEM : 0;
}

int kda_oracle_recurrent(int n_seqs, const int64_t *cu, int H, int dk, int dv,
                         const double *q, const double *k, const double *v, const double *g,
                         const double *beta, const double *init_state, double *o,
                         double *final_state, int n_threads)
{
    problem_t p = {n_seqs, H, dk, dv, cu, q, k, v, g, beta, init_state, o, final_state};
    return run_recurrent(&p, n_threads);
}

/* ------------------------------------------------------------- backward pass ---------- */

/*
 * Reverse sweep of one (sequence, head). Per token, with S_prev the state before it:
 *   forward pieces  Sd = Diag(alpha) S_prev, w = v - Sd^T k, u = beta w, S = Sd + k u^T, o = S^T q
 *   adjoints        dq = S do;  dS += q do^T;  du = dS^T k;  dk = dS u;  dbeta = du . w;
 *                   dv = beta du;  dSd = dS - k (beta du)^T;  dk -= Sd (beta du);
 *                   dg = rowsum(dSd * Sd);  dS_prev = Diag(alpha) dSd
 */
int kda_oracle_backward(int n_seqs, const int64_t *cu, int H, int dk, int dv, const double *q,
                        const double *k, const double *v, const double *g, const double *beta,
                        const double *init_state, const double *d_o, const double *d_final,
                        double *dq, double *dkk, double *dvv, double *dg, double *dbeta,
                        double *d_init)
{
    problem_t p = {n_seqs, H, dk, dv, cu, q, k, v, g, beta, init_state, dq, NULL};
    int err = check_problem(&p);
    if (err) return err;
    if (cu[n_seqs] > cu[0] && (!d_o || !dkk || !dvv || !dg || !dbeta)) return KDA_ORACLE_EBADARG;
    const size_t ss = (size_t)dk * dv;
    for (int n = 0; n < n_seqs; ++n)
        for (int h = 0; h < H; ++h) {
            const int64_t t0 = cu[n], len = cu[n + 1] - cu[n];
            double *hist = malloc(sizeof(double) * (ss * (size_t)(len + 4) + 2 * (size_t)dv));
            if (!hist) return KDA_ORACLE_ENOMEM;
            double *Sd = hist + ss * (size_t)len, *St = Sd + ss, *dS = St + ss, *dSd = dS + ss;
            double *w = dSd + ss, *du = w + dv;
            /* forward: hist[t] = state before token t0 + t */
            load_state(&p, n, h, Sd);
            for (int64_t t = 0; t < len; ++t) {
                size_t r = (size_t)(t0 + t) * H + h;
                memcpy(hist + ss * (size_t)t, Sd, ss * sizeof(double));
                recurrent_token(dk, dv, q + r * dk, k + r * dk, v + r * dv, g + r * dk, beta[r], Sd, St, w);
            }
            if (d_final) memcpy(dS, d_final + ((size_t)n * H + h) * ss, ss * sizeof(double));
            else memset(dS, 0, ss * sizeof(double));
            for (int64_t t = len - 1; t >= 0; --t) {
                size_t r = (size_t)(t0 + t) * H + h;
                const double *kt = k + r * dk, *qt = q + r * dk, *vt = v + r * dv, *gt = g + r * dk;
                const double *dot = d_o + r * dv, bt = beta[r];
                const double *Sp = hist + ss * (size_t)t;
                for (int i = 0; i < dk; ++i) {
                    double a = exp(gt[i]);
                    for (int j = 0; j < dv; ++j) Sd[(size_t)i * dv + j] = a * Sp[(size_t)i * dv + j];
                }
                for (int j = 0; j < dv; ++j) {
                    double kv = 0.0;
                    for (int i = 0; i < dk; ++i) kv += Sd[(size_t)i * dv + j] * kt[i];
                    w[j] = vt[j] - kv;
                }
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) St[(size_t)i * dv + j] = Sd[(size_t)i * dv + j] + kt[i] * bt * w[j];
                /* o = S^T q */
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) acc += St[(size_t)i * dv + j] * dot[j];
                    dq[r * dk + i] = acc;
                }
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) dS[(size_t)i * dv + j] += qt[i] * dot[j];
                /* S = Sd + k u^T */
                double db = 0.0;
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += kt[i] * dS[(size_t)i * dv + j];
                    du[j] = acc;
                    db += acc * w[j];
                }
                dbeta[r] = db;
                for (int j = 0; j < dv; ++j) dvv[r * dv + j] = bt * du[j];
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j)
                        acc += dS[(size_t)i * dv + j] * bt * w[j] - Sd[(size_t)i * dv + j] * bt * du[j];
                    dkk[r * dk + i] = acc;
                }
                /* u = beta (v - Sd^T k): the k-read of Sd */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        dSd[(size_t)i * dv + j] = dS[(size_t)i * dv + j] - kt[i] * bt * du[j];
                /* Sd = Diag(alpha) S_prev */
                for (int i = 0; i < dk; ++i) {
                    double a = exp(gt[i]), acc = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        acc += dSd[(size_t)i * dv + j] * Sd[(size_t)i * dv + j];
                        dS[(size_t)i * dv + j] = a * dSd[(size_t)i * dv + j];
                    }
                    dg[r * dk + i] = acc;
                }
            }
            if (d_init) memcpy(d_init + ((size_t)n * H + h) * ss, dS, ss * sizeof(double));
            free(hist);
        }
    return 0;
}

/* ------------------------------------------------------ literal transition form ------- */

/* S_t = (I - b k k^T) Diag(exp g) S_{t-1} + b k v^T with the transition formed as a matrix. */
int kda_oracle_literal(int n_seqs, const int64_t *cu, int H, int dk, int dv,
                       const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const double *init_state, double *o,
                       double *final_state)
{
    problem_t p = {n_seqs, H, dk, dv, cu, q, k, v, g, beta, init_state, o, final_state};
    int err = check_problem(&p);
    if (err) return err;
    size_t ss = (size_t)dk * dv;
    double *S = malloc(sizeof(double) * (2 * ss + (size_t)dk * dk));
    if (!S) return KDA_ORACLE_ENOMEM;
    double *Sn = S + ss, *M = Sn + ss;
    for (int n = 0; n < n_seqs; ++n)
        for (int h = 0; h < H; ++h) {
            load_state(&p, n, h, S);
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                size_t r = (size_t)t * H + h;
                const double *kt = k + r * dk, *qt = q + r * dk, *vt = v + r * dv, *gt = g + r * dk;
                double bt = beta[r];
                /* M = (I - b k k^T) Diag(alpha) */
                for (int i = 0; i < dk; ++i)
                    for (int c = 0; c < dk; ++c)
                        M[(size_t)i * dk + c] = ((i == c ? 1.0 : 0.0) - bt * kt[i] * kt[c]) * exp(gt[c]);
                /* S_new = M S + b k v^T */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) {
                        double acc = bt * kt[i] * vt[j];
                        for (int c = 0; c < dk; ++c) acc += M[(size_t)i * dk + c] * S[(size_t)c * dv + j];
                        Sn[(size_t)i * dv + j] = acc;
                    }
                memcpy(S, Sn, ss * sizeof(double));
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];
                    o[r * dv + j] = acc;
                }
            }
            store_state(&p, n, h, S);
        }
    free(S);
    return 0;
}

/* ------------------------------------------------------------ chunkwise form ---------- */
/*
 * Per chunk of n <= C tokens with state S at the chunk start (derivation: unroll the
 * recurrence inside the chunk; every intermediate state is Diag(gamma_t) S plus a sum of
 * rank-1 terms k_s u_s^T decayed from s to t):
 *   Gam_r   = sum_{s<=r} g_s               (cumulative log-decay, per key channel)
 *   gam_r   = exp(Gam_r)
 *   Kp = K * gam,  Km = K / gam,  Qp = Q * gam            (element-wise, per channel)
 *   A[r][s] = beta_r <Kp_r, Km_s> for s < r, else 0       (strictly lower)
 *   T       = (I + A)^{-1} Diag(beta)
 *   W = T Kp,  Ut = T V,  U = Ut - W S                      (delta corrections u_s)
 *   O[r]    = Qp_r S + sum_{s<=r} <Qp_r, Km_s> U_s
 *   S_next  = Diag(gam_{n-1}) S + sum_s (K_s * gam_{n-1} / gam_s) U_s^T
 * Optional per-chunk intermediates (each may be NULL) are written for the first (n, h)
 * pair only, chunk after chunk, as fp64 arrays: Gam [n x dk], A [n x n], T [n x n],
 * U [n x dv], S_before [dk x dv] (state at each chunk start).
 */
typedef struct {
    double *Gam, *A, *T, *U, *S_before;
} chunk_dump_t;

static int chunk_one(const problem_t *p, int C, int n, int h, double *ws, chunk_dump_t *dump)
{
    const int H = p->H, dk = p->dk, dv = p->dv;
    double *S = ws;                          /* dk*dv */
    double *Gam = S + (size_t)dk * dv;       /* C*dk  */
    double *gam = Gam + (size_t)C * dk;      /* C*dk  */
    double *Kp = gam + (size_t)C * dk;       /* C*dk  */
    double *Km = Kp + (size_t)C * dk;        /* C*dk  */
    double *Qp = Km + (size_t)C * dk;        /* C*dk  */
    double *A = Qp + (size_t)C * dk;         /* C*C   */
    double *X = A + (size_t)C * C;           /* C*C   */
    double *T = X + (size_t)C * C;           /* C*C   */
    double *W = T + (size_t)C * C;           /* C*dk  */
    double *U = W + (size_t)C * dk;          /* C*dv  */
    double *Sn = U + (size_t)C * dv;         /* dk*dv */
    size_t off_G = 0, off_A = 0, off_U = 0, off_S = 0;

    load_state(p, n, h, S);
    for (int64_t c0 = p->cu[n]; c0 < p->cu[n + 1]; c0 += C) {
        int len = (int)((p->cu[n + 1] - c0) < C ? (p->cu[n + 1] - c0) : C);
#define ROW(t) ((size_t)(c0 + (t)) * H + h)
        for (int i = 0; i < dk; ++i) {
            double run = 0.0;
            for (int r = 0; r < len; ++r) {
                run += p->g[ROW(r) * dk + i];
                Gam[(size_t)r * dk + i] = run;
                gam[(size_t)r * dk + i] = exp(run);
            }
        }
        for (int r = 0; r < len; ++r)
            for (int i = 0; i < dk; ++i) {
                double kk = p->k[ROW(r) * dk + i], qq = p->q[ROW(r) * dk + i], e = gam[(size_t)r * dk + i];
                Kp[(size_t)r * dk + i] = kk * e;
                Km[(size_t)r * dk + i] = kk / e;
                Qp[(size_t)r * dk + i] = qq * e;
            }
        for (int r = 0; r < len; ++r)
            for (int s = 0; s < len; ++s) {
                double acc = 0.0;
                if (s < r)
                    for (int i = 0; i < dk; ++i) acc += Kp[(size_t)r * dk + i] * Km[(size_t)s * dk + i];
                A[(size_t)r * len + s] = s < r ? p->beta[ROW(r)] * acc : 0.0;
            }
        /* X = (I + A)^{-1}: forward substitution, one unit column at a time. */
        for (int col = 0; col < len; ++col)
            for (int r = 0; r < len; ++r) {
                double x = (r == col) ? 1.0 : 0.0;
                for (int s = 0; s < r; ++s) x -= A[(size_t)r * len + s] * X[(size_t)s * len + col];
                X[(size_t)r * len + col] = x;
            }
        for (int r = 0; r < len; ++r)
            for (int s = 0; s < len; ++s) T[(size_t)r * len + s] = X[(size_t)r * len + s] * p->beta[ROW(s)];
        /* W = T Kp ; U = T V - W S */
        for (int r = 0; r < len; ++r) {
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int s = 0; s < len; ++s) acc += T[(size_t)r * len + s] * Kp[(size_t)s * dk + i];
                W[(size_t)r * dk + i] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                double tv = 0.0, ws_ = 0.0;
                for (int s = 0; s < len; ++s) tv += T[(size_t)r * len + s] * p->v[ROW(s) * dv + j];
                for (int i = 0; i < dk; ++i) ws_ += W[(size_t)r * dk + i] * S[(size_t)i * dv + j];
                U[(size_t)r * dv + j] = tv - ws_;
            }
        }
        /* O = Qp S + tril_0(Qp Km^T) U */
        for (int r = 0; r < len; ++r)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += Qp[(size_t)r * dk + i] * S[(size_t)i * dv + j];
                for (int s = 0; s <= r; ++s) {
                    double qk = 0.0;
                    for (int i = 0; i < dk; ++i) qk += Qp[(size_t)r * dk + i] * Km[(size_t)s * dk + i];
                    acc += qk * U[(size_t)s * dv + j];
                }
                p->o[ROW(r) * dv + j] = acc;
            }
        if (dump) {
            if (dump->Gam) memcpy(dump->Gam + off_G, Gam, sizeof(double) * (size_t)len * dk);
            if (dump->A) memcpy(dump->A + off_A, A, sizeof(double) * (size_t)len * len);
            if (dump->T) memcpy(dump->T + off_A, T, sizeof(double) * (size_t)len * len);
            if (dump->U) memcpy(dump->U + off_U, U, sizeof(double) * (size_t)len * dv);
            if (dump->S_before) memcpy(dump->S_before + off_S, S, sizeof(double) * (size_t)dk * dv);
            off_G += (size_t)len * dk; off_A += (size_t)len * len; off_U += (size_t)len * dv;
            off_S += (size_t)dk * dv;
        }
        /* S_next = Diag(gam_last) S + sum_s (K_s * gam_last / gam_s) U_s^T */
        const double *glast = gam + (size_t)(len - 1) * dk;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                double acc = glast[i] * S[(size_t)i * dv + j];
                for (int s = 0; s < len; ++s)
                    acc += p->k[ROW(s) * dk + i] * glast[i] / gam[(size_t)s * dk + i] * U[(size_t)s * dv + j];
                Sn[(size_t)i * dv + j] = acc;
            }
        memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
#undef ROW
    }
    store_state(p, n, h, S);
    return 0;
}

int kda_oracle_chunked(int n_seqs, const int64_t *cu, int H, int dk, int dv, int C,
                       const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const double *init_state, double *o,
                       double *final_state, int n_threads,
                       double *dump_Gam, double *dump_A, double *dump_T, double *dump_U,
                       double *dump_S_before)
{
    problem_t p = {n_seqs, H, dk, dv, cu, q, k, v, g, beta, init_state, o, final_state};
    int err = check_problem(&p);
    if (err) return err;
    if (C <= 0) return KDA_ORACLE_EBADARG;
    size_t ws_elems = 2 * (size_t)dk * dv + 6 * (size_t)C * dk + 3 * (size_t)C * C + (size_t)C * dv;
    chunk_dump_t dump = {dump_Gam, dump_A, dump_T, dump_U, dump_S_before};
    int want_dump = dump_Gam || dump_A || dump_T || dump_U || dump_S_before;
    const int pairs = n_seqs * H;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int ph = 0; ph < pairs; ++ph) {
        double *ws = malloc(sizeof(double) * ws_elems);
        if (!ws) { failed |= 1; continue; }
        chunk_one(&p, C, ph / H, ph % H, ws, (want_dump && ph == 0) ? &dump : NULL);
        free(ws);
    }
    return failed ? KDA_ORACLE_ENOMEM : 0;
}

int kda_oracle_scaled_sigmoid_gate(int64_t n, const double *x, double bound, double *g)
{
    if (n < 0 || !x || !g || !(bound > 0.0)) return -1;
    for (int64_t i = 0; i < n; ++i) {
        const double sig = 1.0 / (1.0 + exp(-x[i]));  /* the logistic function */
        g[i] = -bound * sig;
    }
    return 0;
}

int kda_oracle_l2_normalize(int64_t rows, int64_t d, const double *x, double eps, double *y)
{
    if (rows < 0 || d <= 0 || !x || !y || !(eps >= 0.0)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t i = 0; i < d; ++i) ss += x[r * d + i] * x[r * d + i];
        const double norm = sqrt(ss + eps);
        for (int64_t i = 0; i < d; ++i) y[r * d + i] = norm > 0.0 ? x[r * d + i] / norm : 0.0;
    }
    return 0;
}

int kda_oracle_output_gate(int64_t n, const double *o, const double *z, double *y)
{
    if (n < 0 || !o || !z || !y) return -1;
    for (int64_t i = 0; i < n; ++i) y[i] = o[i] / (1.0 + exp(-z[i]));
    return 0;
}

int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
